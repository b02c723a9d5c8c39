// moe_api.cu -- the C ABI declared in include/moe.h: context, workspace and
// the launch sequence of the MoE layer.
#include <stdlib.h>
#include <string.h>

#include <array>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/moe.h"
#include "kernels.h"

using namespace moe;

struct moe_ctx {
    int d = 0, F = 0, n = 0, k = 0;
    int dtype = MOE_BF16;
    const float* bias = nullptr;
    int decode_max_t = 128;     // weight streaming beats the grouped GEMMs up to here (T=128: 516 vs 534 us/layer)
    long long wait_limit_us = 2000000;
    int force_path = 0;
    int gemm_pair = 0;          // 0 auto, 1 single CTA, 2 CTA pairs
    int host_out = 1;           // moe_forward_host: 1 = kernels write y into pinned host memory directly
    int fp8_widen = 0;          // moe_forward_fp8: 0 = e4m3 MMA on split token rows, 1 = weights widened to bf16
    int decode_streamk = 1;     // bf16 weight streaming: 1 = stream-K split of K, 0 = uniform splits
    int device = 0;
    int num_sms = 148;
    int* status_host = nullptr;   // host-mapped
    int* status_dev = nullptr;    // device alias
    // workspace (one allocation)
    int cap_T = -1;
    int cap_dec = 0;            // tokens the decode partial-sum buffers hold
    void* ws = nullptr;
    size_t ws_bytes = 0;
    int32_t* topk_idx = nullptr;
    float* topk_w = nullptr;
    int32_t* perm = nullptr;
    int32_t* inv = nullptr;
    int* sched = nullptr;
    int* xchg = nullptr;        // grid-barrier words and block counts of the fused routing kernel
    int* ccnt = nullptr;        // [T][d/128] arrival counters of the combine fused into the W2 epilogue
    float* rstd = nullptr;      // [T] 1/rms of each row (residual blocks: RMSNorm before routing)
    void* Xp = nullptr;
    void* H = nullptr;
    float* Ys = nullptr;
    void* xbuf = nullptr;
    void* xbuf2 = nullptr;      // moe_forward_host stages x in xbuf / xbuf2 on alternate calls
    void* ybuf = nullptr;
    // moe_forward_host: input copies on a stream of their own, overlapping the previous call
    cudaStream_t h2d_stream = nullptr;
    cudaEvent_t ev_h2d[2] = {nullptr, nullptr};
    cudaEvent_t ev_xfree[2] = {nullptr, nullptr};
    int host_slot = 0;
    float* Pa = nullptr;        // decode partial sums [S][R][F] (W1 rows), [S][R][F] (W3 rows)
    float* Pb = nullptr;
    float* P2 = nullptr;        // decode partial sums [S][R][d] (W2 rows)
    uint8_t* Xq = nullptr;      // e4m3 MMA path: hi/lo e4m3 token rows [2R][d] and SwiGLU rows [2R][F],
    uint8_t* Hq = nullptr;      //   with 1/scale per row
    float* xinv = nullptr;
    float* hinv = nullptr;
    CUtensorMap map_Xp, map_H, map_Xp32, map_H32;
    bool maps_ok = false;
    // per-stage CUDA-event timing (MOE_OPT_STAGE_TIMING)
    bool stage_timing = false;
    std::vector<cudaEvent_t> ev_free;
    std::vector<std::array<cudaEvent_t, 5>> ev_calls;
};

namespace {

size_t esize(int dtype) { return dtype == MOE_F32 ? 4 : 2; }
size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

struct Layout {
    size_t topk_idx, topk_w, perm, inv, sched, xchg, ccnt, rstd, Xp, H, Ys, xbuf, xbuf2, ybuf, Pa, Pb, P2, Xq, Hq, xinv,
        hinv, total;
};

Layout layout_for(const moe_ctx* c, int T, int Tdec) {
    Layout L{};
    const size_t R = static_cast<size_t>(c->k) * static_cast<size_t>(T > 0 ? T : 1);
    const size_t Tn = static_cast<size_t>(T > 0 ? T : 1);
    const size_t es = esize(c->dtype);
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off += align256(bytes); return o; };
    L.topk_idx = take(R * 4);
    L.topk_w = take(R * 4);
    L.perm = take(R * 4);
    L.inv = take(R * 4);
    L.sched = take(static_cast<size_t>(sched_ints(c->n)) * 4);
    L.xchg = take(static_cast<size_t>(fused_route_xchg_ints()) * 4);
    L.ccnt = take(Tn * static_cast<size_t>((c->d + 127) / 128) * 4);
    L.rstd = take(Tn * 4);
    L.Xp = take(R * c->d * es);
    L.H = take(R * c->F * es);
    L.Ys = take(R * c->d * 4);
    L.xbuf = take(Tn * c->d * es);
    L.xbuf2 = take(Tn * c->d * es);
    L.ybuf = take(Tn * c->d * es);
    const size_t Rd = static_cast<size_t>(c->k) * static_cast<size_t>(Tdec > 0 ? Tdec : 0);
    L.Pa = take(kDecodeMaxSplits * Rd * c->F * 4);
    L.Pb = take(kDecodeMaxSplits * Rd * c->F * 4);
    L.P2 = take(kDecodeMaxSplits * Rd * c->d * 4);
    L.Xq = take(c->dtype == MOE_BF16 ? 2 * Rd * c->d : 0);
    L.Hq = take(c->dtype == MOE_BF16 ? 2 * Rd * c->F : 0);
    L.xinv = take(Rd * 4);
    L.hinv = take(kDecodeMaxSplits * Rd * 4);
    L.total = off;
    return L;
}

KStatus kstatus(const moe_ctx* c) {
    KStatus st;
    st.word = c->status_dev;
    st.wait_ns = static_cast<uint64_t>(c->wait_limit_us) * 1000ull;
    return st;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_fail(cudaError_t e) { return e == cudaErrorMemoryAllocation ? MOE_ERR_OOM : MOE_ERR_CUDA; }

bool env_flag(const char* name) {
    const char* v = getenv(name);
    return v && *v && strcmp(v, "0") != 0;
}

// Make sure the workspace holds T tokens (and, for the decode kernels, their
// partial sums).  Growth frees the old buffer after synchronising the stream;
// it is refused while the stream is being captured.
int ensure_workspace(moe_ctx* c, int T, cudaStream_t s, bool decode = false) {
    if (T <= c->cap_T && c->ws && (!decode || T <= c->cap_dec)) return MOE_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone) return MOE_ERR_INVALID;
    if (env_flag("MOE_FAIL_WORKSPACE_ALLOC")) return MOE_ERR_OOM;   // host-side fault injection for tests
    int Tdec = decode ? T : 0;
    if (Tdec > kDecodeMaxT) Tdec = kDecodeMaxT;
    if (c->ws && c->cap_dec > Tdec) Tdec = c->cap_dec;
    if (c->ws && c->cap_T > T) T = c->cap_T;
    Layout L = layout_for(c, T, Tdec);
    if (c->ws) {
        cudaStreamSynchronize(s);
        cudaDeviceSynchronize();
        cudaFree(c->ws);
        c->ws = nullptr;
        c->cap_T = -1;
        c->cap_dec = 0;
        c->maps_ok = false;
    }
    void* p = nullptr;
    cudaError_t e = cudaMalloc(&p, L.total);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_OOM;
    }
    char* b = static_cast<char*>(p);
    c->ws = p;
    c->ws_bytes = L.total;
    c->topk_idx = reinterpret_cast<int32_t*>(b + L.topk_idx);
    c->topk_w = reinterpret_cast<float*>(b + L.topk_w);
    c->perm = reinterpret_cast<int32_t*>(b + L.perm);
    c->inv = reinterpret_cast<int32_t*>(b + L.inv);
    c->sched = reinterpret_cast<int*>(b + L.sched);
    c->xchg = reinterpret_cast<int*>(b + L.xchg);
    c->ccnt = reinterpret_cast<int*>(b + L.ccnt);
    c->rstd = reinterpret_cast<float*>(b + L.rstd);
    c->Xp = b + L.Xp;
    c->H = b + L.H;
    c->Ys = reinterpret_cast<float*>(b + L.Ys);
    c->xbuf = b + L.xbuf;
    c->xbuf2 = b + L.xbuf2;
    c->ybuf = b + L.ybuf;
    c->Pa = reinterpret_cast<float*>(b + L.Pa);
    c->Pb = reinterpret_cast<float*>(b + L.Pb);
    c->P2 = reinterpret_cast<float*>(b + L.P2);
    c->Xq = reinterpret_cast<uint8_t*>(b + L.Xq);
    c->Hq = reinterpret_cast<uint8_t*>(b + L.Hq);
    c->xinv = reinterpret_cast<float*>(b + L.xinv);
    c->hinv = reinterpret_cast<float*>(b + L.hinv);
    c->cap_T = T;
    c->cap_dec = Tdec;
    if (cudaMemsetAsync(c->xchg, 0, L.rstd - L.xchg, s) != cudaSuccess) return MOE_ERR_CUDA;   // every counter region
    // Tensor maps of the workspace activations cover the full capacity; rows
    // beyond the live K*T are never valid rows of any tile.
    if (c->dtype == MOE_BF16) {
        const uint64_t R = static_cast<uint64_t>(c->k) * static_cast<uint64_t>(T > 0 ? T : 1);
        c->maps_ok = encode_map_bf16_2d(&c->map_Xp, c->Xp, R, c->d, 128) &&
                     encode_map_bf16_2d(&c->map_H, c->H, R, c->F, 128) &&
                     encode_map_bf16_2d(&c->map_Xp32, c->Xp, R, c->d, 32) &&
                     encode_map_bf16_2d(&c->map_H32, c->H, R, c->F, 32);
        if (!c->maps_ok) return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

bool tc_shape_ok(const moe_ctx* c) { return c->d % 256 == 0 && c->F % 128 == 0; }

// Device address of pinned, mapped host memory (pinned allocations are mapped
// on every 64-bit system with unified addressing), or null for anything else.
void* mapped_host_alias(void* p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost || !a.devicePointer) return nullptr;
    return a.devicePointer;
}

// The input-copy stream and its events (created on first use).
bool ensure_copy_stream(moe_ctx* c) {
    if (c->h2d_stream) return true;
    cudaStream_t st = nullptr;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return false;
    for (int i = 0; i < 2; ++i) {
        if (cudaEventCreateWithFlags(&c->ev_h2d[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&c->ev_xfree[i], cudaEventDisableTiming) != cudaSuccess) {
            cudaStreamDestroy(st);
            return false;
        }
    }
    c->h2d_stream = st;
    return true;
}

// The weight-streaming kernels serve bf16 batches of up to decode_max_t tokens.
bool use_decode(const moe_ctx* c, int T) {
    if (c->dtype != MOE_BF16 || c->n > 31 || T > kDecodeMaxT || c->force_path == 1) return false;
    return c->force_path == 2 || T <= c->decode_max_t;
}

// Which grouped GEMMs run on CTA pairs.  Pairs move a third fewer operand
// bytes per FLOP.  At the Mixtral shape, timed in windows of 5-20 calls
// alternating with single CTAs, a layer with both GEMMs on pairs was 1.5-4.5%
// faster at T = 4096, ~3% at T = 8192 and ~1.5% on the skewed T = 32768 batch;
// in 400-call runs at the board's power cap, 1.3% faster.  So by default both
// run on pairs when the device can co-schedule them (1 forces single CTAs).
bool use_pair13(const moe_ctx* c) { return c->gemm_pair != 1 && pair_gemm_available(c->num_sms); }
bool use_pair2(const moe_ctx* c) { return c->gemm_pair != 1 && pair_gemm_available(c->num_sms); }

// Stages of one forward call, in launch order.
constexpr int kStages = 4;
const char* const kStageNames[kStages] = {"route", "expert_w1w3_swiglu", "expert_w2_gate", "combine"};

// Stage boundaries of the current call: an NVTX range for the call and, inside
// it, one per stage, on the host thread that launches them; CUDA events on the
// call's stream when stage timing is on.
struct StageMarks {
    moe_ctx* c = nullptr;
    cudaStream_t s = nullptr;
    std::array<cudaEvent_t, kStages + 1> ev{};
    bool on = false;
    int next = 0;             // events ev[0 .. next) recorded
    bool range_open = false;
    StageMarks(moe_ctx* ctx, cudaStream_t st, const char* call = "moe_forward") : c(ctx), s(st) {
        nvtxRangePushA(call);
        if (!c->stage_timing) return;
        for (int i = 0; i <= kStages; ++i) {
            if (!c->ev_free.empty()) {
                ev[i] = c->ev_free.back();
                c->ev_free.pop_back();
            } else if (cudaEventCreate(&ev[i]) != cudaSuccess) {
                for (int j = 0; j < i; ++j) c->ev_free.push_back(ev[j]);
                return;
            }
        }
        on = true;
        cudaEventRecord(ev[0], s);
        next = 1;
    }
    // The launches from here on belong to stage i.
    void begin(int i) {
        if (range_open) nvtxRangePop();
        nvtxRangePushA(kStageNames[i]);
        range_open = true;
        if (on)
            while (next <= i) cudaEventRecord(ev[next++], s);
    }
    void finish() {
        if (range_open) {
            nvtxRangePop();
            range_open = false;
        }
        if (on) {
            while (next <= kStages) cudaEventRecord(ev[next++], s);
            c->ev_calls.push_back(ev);
            on = false;
        }
    }
    ~StageMarks() {
        if (range_open) nvtxRangePop();
        nvtxRangePop();
        if (on)
            for (int i = 0; i <= kStages; ++i) c->ev_free.push_back(ev[i]);
    }
};

// router + top-k + dispatch (+ the row gather into Xp when gather is set);
// norm_eps >= 0: RMSNorm the rows first
int run_route(moe_ctx* c, const void* x, const float* Wg, int T, cudaStream_t s, float* logits, bool gather,
              float norm_eps = -1.0f) {
    const ElemType et = c->dtype == MOE_F32 ? ElemType::F32 : ElemType::BF16;
    cudaError_t e = launch_fused_route(et, x, Wg, c->bias, T, c->d, c->n, c->k, c->topk_idx, c->topk_w, logits,
                                       c->sched, c->perm, c->inv, gather ? c->Xp : nullptr, c->xchg,
                                       norm_eps, norm_eps >= 0.0f ? c->rstd : nullptr, kstatus(c), c->num_sms, s);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

// y = MoE(x); with norm_eps >= 0 and resid: y = resid + MoE(RMSNorm(x)) (the
// residual block of a stack, x == resid == y allowed).
int run_forward(moe_ctx* c, const void* x, const float* Wg, const void* W1, const void* W3, const void* W2, void* y,
                int T, cudaStream_t s, float norm_eps = -1.0f, const void* resid = nullptr) {
    const ElemType et = c->dtype == MOE_F32 ? ElemType::F32 : ElemType::BF16;
    const int R = c->k * T;
    StageMarks marks(c, s);
    marks.begin(0);
    int rc = run_route(c, x, Wg, T, s, nullptr, true, norm_eps);
    if (rc != MOE_OK) return rc;
    cudaError_t e = cudaSuccess;
    if (et == ElemType::F32) {
        marks.begin(1);
        e = launch_simt_gemm13(et, c->Xp, W1, W3, c->H, c->sched, c->n, c->d, c->F, R, s);
        if (e != cudaSuccess) return cuda_fail(e);
        marks.begin(2);
        e = launch_simt_gemm2(et, c->H, W2, c->Ys, c->sched, c->perm, c->topk_w, c->n, c->d, c->F, R, s);
        if (e != cudaSuccess) return cuda_fail(e);
    } else if (use_decode(c, T)) {
        CUtensorMap mW1, mW3, mW2;
        const uint64_t nF = static_cast<uint64_t>(c->n) * c->F, nd = static_cast<uint64_t>(c->n) * c->d;
        if (!encode_map_bf16_2d(&mW1, W1, nF, c->d, 128) || !encode_map_bf16_2d(&mW3, W3, nF, c->d, 128) ||
            !encode_map_bf16_2d(&mW2, W2, nd, c->F, 128))
            return MOE_ERR_CUDA;
        const KStatus st = kstatus(c);
        const int touched = c->n < R ? c->n : R;
        // uniform K splits, or 0: stream-K (SplitGeom in kernels.h).  Stream-K from two
        // tokens on: measured 2-13 us faster per layer at T = 8..128, ~2 us slower at T = 1.
        const bool sk = c->decode_streamk && T > 1;
        const int s0 = sk ? 0 : decode_pick_splits(touched * (c->F / 128), c->d / 64, c->num_sms);
        const int s1 = sk ? 0 : decode_pick_splits(touched * (c->d / 128), c->F / 64, c->num_sms);
        marks.begin(1);
        int* ready = c->xchg + kReadyWord;
        e = launch_decode_w13(mW1, mW3, c->map_Xp32, c->sched, c->n, c->d, c->F, T, c->k, s0, c->Pa, c->Pb, st,
                              c->num_sms, s, ready);
        if (e != cudaSuccess) return cuda_fail(e);
        const SplitGeom g13 = decode_geom(s0, c->d / 64, c->F / 128, c->sched, c->n, c->num_sms);
        e = launch_decode_swiglu(c->Pa, c->Pb, g13, R, c->F, static_cast<__nv_bfloat16*>(c->H), s);
        if (e != cudaSuccess) return cuda_fail(e);
        marks.begin(2);
        e = launch_decode_w2(mW2, c->map_H32, c->sched, c->n, c->d, c->F, T, c->k, s1, c->P2, st, c->num_sms, s,
                             ready);
        if (e != cudaSuccess) return cuda_fail(e);
        marks.begin(3);
        const SplitGeom g2 = decode_geom(s1, c->F / 64, c->d / 128, c->sched, c->n, c->num_sms);
        e = launch_decode_combine(et, c->P2, g2, R, c->inv, c->topk_idx, c->topk_w, T, c->k, c->d, resid, y, s);
        if (e != cudaSuccess) return cuda_fail(e);
        marks.finish();
        return MOE_OK;
    } else {
        const bool pair13 = use_pair13(c), pair2 = use_pair2(c);
        if (c->gemm_pair == 2 && !pair13) return MOE_ERR_UNSUPPORTED;
        CUtensorMap mW1, mW3, mW2;
        const uint64_t nF = static_cast<uint64_t>(c->n) * c->F, nd = static_cast<uint64_t>(c->n) * c->d;
        if (!encode_map_bf16_2d(&mW1, W1, nF, c->d, 128) || !encode_map_bf16_2d(&mW3, W3, nF, c->d, 128) ||
            !encode_map_bf16_2d(&mW2, W2, nd, c->F, pair2 ? 128 : 256))
            return MOE_ERR_CUDA;
        const KStatus st = kstatus(c);
        CUtensorMap mW1h, mW3h;
        if (pair13 && (!encode_map_bf16_2d(&mW1h, W1, nF, c->d, 64) || !encode_map_bf16_2d(&mW3h, W3, nF, c->d, 64)))
            return MOE_ERR_CUDA;
        marks.begin(1);
        if (pair13)
            e = launch_pair_gemm13(c->map_Xp, mW1, mW3, mW1h, mW3h, c->sched, c->n, c->d, c->F, R,
                                   static_cast<__nv_bfloat16*>(c->H), st, c->num_sms, s);
        else
            e = launch_tc_gemm13(c->map_Xp, mW1, mW3, c->sched, c->n, c->d, c->F, R,
                                 static_cast<__nv_bfloat16*>(c->H), st, c->num_sms, s);
        if (e != cudaSuccess) return cuda_fail(e);
        CombineArgs comb{};
        comb.cnt = c->ccnt;
        comb.y = static_cast<__nv_bfloat16*>(y);
        comb.resid = static_cast<const __nv_bfloat16*>(resid);
        comb.K = c->k;
        comb.nblk = c->d / 128;
        comb.d = c->d;
        marks.begin(2);
        if (pair2)
            e = launch_pair_gemm2(c->map_H, mW2, c->sched, c->n, c->d, c->F, R, c->Ys, c->perm, c->topk_w, comb, st,
                                  c->num_sms, s);
        else
            e = launch_tc_gemm2(c->map_H, mW2, c->sched, c->n, c->d, c->F, R, c->Ys, c->perm, c->topk_w, comb, st,
                                c->num_sms, s);
        if (e != cudaSuccess) return cuda_fail(e);
        marks.begin(3);   // the combine ran inside the W2 epilogue
        marks.finish();
        return MOE_OK;
    }
    marks.begin(3);
    e = launch_combine(et, c->Ys, T, c->k, c->d, resid, y, s);
    if (e != cudaSuccess) return cuda_fail(e);
    marks.finish();
    return MOE_OK;
}

// y = MoE(x) for T <= kDecodeMaxT tokens with e4m3 expert weights and fp32
// row scales: the weight-streaming path, same split choice and combine kernel
// as the bf16 one.  By default the weights meet the tokens in the e4m3 MMA
// (token rows split into hi/lo e4m3 rows, decode_fp8_mma.cu); with
// MOE_OPT_FP8_WIDEN the weights are widened to bf16 on chip (decode_fp8.cu).
int run_forward_fp8(moe_ctx* c, const void* x, const float* Wg, const uint8_t* W1q, const float* W1s,
                    const uint8_t* W3q, const float* W3s, const uint8_t* W2q, const float* W2s, void* y, int T,
                    cudaStream_t s) {
    const int R = c->k * T;
    StageMarks marks(c, s, "moe_forward_fp8");
    marks.begin(0);
    int rc = run_route(c, x, Wg, T, s, nullptr, true);
    if (rc != MOE_OK) return rc;
    CUtensorMap mW1, mW3, mW2;
    const uint64_t nF = static_cast<uint64_t>(c->n) * c->F, nd = static_cast<uint64_t>(c->n) * c->d;
    const KStatus st = kstatus(c);
    const int touched = c->n < R ? c->n : R;
    cudaError_t e = cudaSuccess;
    int s1 = 1;
    if (!c->fp8_widen) {
        CUtensorMap mXq, mHq;
        if (!encode_map_u8_sw128(&mW1, W1q, nF, c->d, 128) || !encode_map_u8_sw128(&mW3, W3q, nF, c->d, 128) ||
            !encode_map_u8_sw128(&mW2, W2q, nd, c->F, 128) ||
            !encode_map_u8_sw128(&mXq, c->Xq, 2ull * R, c->d, 32) || !encode_map_u8_sw128(&mHq, c->Hq, 2ull * R, c->F, 32))
            return MOE_ERR_CUDA;
        const int s0 = decode_pick_splits(touched * (c->F / 128), c->d / 128, c->num_sms);
        s1 = decode_pick_splits(touched * (c->d / 128), c->F / 128, c->num_sms);
        marks.begin(1);
        e = launch_split_rows_e4m3(static_cast<const __nv_bfloat16*>(c->Xp), R, c->d, c->Xq, c->xinv, s);
        if (e == cudaSuccess)
            e = launch_decode_f8_w13(mW1, mW3, mXq, W1s, W3s, c->xinv, c->sched, c->n, c->d, c->F, T, c->k, s0, c->Pa,
                                     c->Pb, st, c->num_sms, s);
        if (e == cudaSuccess) e = launch_decode_swiglu_split(c->Pa, c->Pb, s0, R, c->F, s1, c->Hq, c->hinv, s);
        if (e != cudaSuccess) return cuda_fail(e);
        marks.begin(2);
        e = launch_decode_f8_w2(mW2, mHq, W2s, c->hinv, c->sched, c->n, c->d, c->F, T, c->k, s1, c->P2, st,
                                c->num_sms, s);
        if (e != cudaSuccess) return cuda_fail(e);
    } else {
        if (!encode_map_u8_sw64(&mW1, W1q, nF, c->d) || !encode_map_u8_sw64(&mW3, W3q, nF, c->d) ||
            !encode_map_u8_sw64(&mW2, W2q, nd, c->F))
            return MOE_ERR_CUDA;
        const int s0 = decode_pick_splits(touched * (c->F / 128), c->d / 64, c->num_sms);
        s1 = decode_pick_splits(touched * (c->d / 128), c->F / 64, c->num_sms);
        marks.begin(1);
        e = launch_decode_fp8_w13(mW1, mW3, c->map_Xp32, W1s, W3s, c->sched, c->n, c->d, c->F, T, c->k, s0, c->Pa,
                                  c->Pb, st, c->num_sms, s);
        if (e == cudaSuccess)
            e = launch_decode_swiglu(c->Pa, c->Pb, decode_geom(s0, c->d / 64, c->F / 128, c->sched, c->n, c->num_sms),
                                     R, c->F, static_cast<__nv_bfloat16*>(c->H), s);
        if (e != cudaSuccess) return cuda_fail(e);
        marks.begin(2);
        e = launch_decode_fp8_w2(mW2, c->map_H32, W2s, c->sched, c->n, c->d, c->F, T, c->k, s1, c->P2, st,
                                 c->num_sms, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    marks.begin(3);
    e = launch_decode_combine(ElemType::BF16, c->P2, decode_geom(s1, 1, c->d / 128, c->sched, c->n, c->num_sms), R,
                              c->inv, c->topk_idx, c->topk_w, T, c->k, c->d, nullptr, y, s);
    if (e != cudaSuccess) return cuda_fail(e);
    marks.finish();
    return MOE_OK;
}

}  // namespace

extern "C" {

moe_ctx* moe_create(int d, int d_ff, int n_experts, int k) {
    if (d <= 0 || d % 8 != 0 || d_ff <= 0 || n_experts < 1 || n_experts > 32 || k < 1 || k > n_experts) return nullptr;
    // the router stages W_g [n][d] fp32 in shared memory
    if (static_cast<size_t>(n_experts) * d * 4 > 200 * 1024) return nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    moe_ctx* c = new moe_ctx();
    c->d = d;
    c->F = d_ff;
    c->n = n_experts;
    c->k = k;
    c->device = dev;
    cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (c->num_sms <= 0) c->num_sms = 148;
    if (const char* v = getenv("MOE_WAIT_LIMIT_US")) c->wait_limit_us = atoll(v) > 0 ? atoll(v) : c->wait_limit_us;
    if (cudaHostAlloc(reinterpret_cast<void**>(&c->status_host), sizeof(int), cudaHostAllocMapped) != cudaSuccess ||
        cudaHostGetDevicePointer(reinterpret_cast<void**>(&c->status_dev), c->status_host, 0) != cudaSuccess) {
        cudaGetLastError();
        if (c->status_host) cudaFreeHost(c->status_host);
        delete c;
        return nullptr;
    }
    *c->status_host = 0;
    return c;
}

int moe_set_dtype(moe_ctx* c, int dtype) {
    if (!c || (dtype != MOE_BF16 && dtype != MOE_F32)) return MOE_ERR_INVALID;
    if (dtype != c->dtype) {
        if (c->ws) {
            cudaDeviceSynchronize();
            cudaFree(c->ws);
            c->ws = nullptr;
            c->cap_T = -1;
            c->cap_dec = 0;
            c->maps_ok = false;
        }
        c->dtype = dtype;
    }
    return MOE_OK;
}

int moe_set_router_bias(moe_ctx* c, const float* b) {
    if (!c) return MOE_ERR_INVALID;
    if (b && !aligned16(b)) return MOE_ERR_INVALID;
    c->bias = b;
    return MOE_OK;
}

int moe_set_option(moe_ctx* c, int option, long long value) {
    if (!c) return MOE_ERR_INVALID;
    switch (option) {
        case MOE_OPT_DECODE_MAX_T:
            if (value < 0) return MOE_ERR_INVALID;
            c->decode_max_t = static_cast<int>(value);
            return MOE_OK;
        case MOE_OPT_WAIT_LIMIT_US:
            if (value <= 0) return MOE_ERR_INVALID;
            c->wait_limit_us = value;
            return MOE_OK;
        case MOE_OPT_FORCE_PATH:
            if (value < 0 || value > 2) return MOE_ERR_INVALID;
            c->force_path = static_cast<int>(value);
            return MOE_OK;
        case MOE_OPT_HOST_OUTPUT:
            if (value < 0 || value > 1) return MOE_ERR_INVALID;
            c->host_out = static_cast<int>(value);
            return MOE_OK;
        case MOE_OPT_GEMM_PAIR:
            if (value < 0 || value > 2) return MOE_ERR_INVALID;
            c->gemm_pair = static_cast<int>(value);
            return MOE_OK;
        case MOE_OPT_STAGE_TIMING:
            if (value < 0 || value > 1) return MOE_ERR_INVALID;
            c->stage_timing = value != 0;
            return MOE_OK;
        case MOE_OPT_FP8_WIDEN:
            if (value < 0 || value > 1) return MOE_ERR_INVALID;
            c->fp8_widen = static_cast<int>(value);
            return MOE_OK;
        case MOE_OPT_DECODE_STREAMK:
            if (value < 0 || value > 1) return MOE_ERR_INVALID;
            c->decode_streamk = static_cast<int>(value);
            return MOE_OK;
        default:
            return MOE_ERR_INVALID;
    }
}

size_t moe_workspace_bytes(const moe_ctx* c, int T) {
    if (!c || T < 0) return 0;
    int Tdec = T < c->decode_max_t ? T : c->decode_max_t;
    if (Tdec > kDecodeMaxT) Tdec = kDecodeMaxT;
    return layout_for(c, T, c->dtype == MOE_BF16 ? Tdec : 0).total;
}

int moe_reserve(moe_ctx* c, int T_max) {
    if (!c || T_max < 0) return MOE_ERR_INVALID;
    int Tdec = T_max < c->decode_max_t ? T_max : c->decode_max_t;
    if (Tdec > kDecodeMaxT) Tdec = kDecodeMaxT;
    int rc = ensure_workspace(c, T_max, nullptr, false);
    if (rc == MOE_OK && c->dtype == MOE_BF16 && Tdec > 0) rc = ensure_workspace(c, Tdec, nullptr, true);
    return rc;
}

int moe_route(moe_ctx* c, const void* x, const float* Wg, int T, int32_t* topk_idx, float* topk_w, int32_t* counts,
              int32_t* offsets, int32_t* perm, moe_stream_t stream) {
    if (!c || T < 0) return MOE_ERR_INVALID;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (T > 0 && (!x || !Wg || !aligned16(x) || !aligned16(Wg))) return MOE_ERR_INVALID;
    int rc = ensure_workspace(c, T, s);
    if (rc != MOE_OK) return rc;
    if (T > 0) {
        rc = run_route(c, x, Wg, T, s, nullptr, false);
        if (rc != MOE_OK) return rc;
    } else {
        if (cudaMemsetAsync(c->sched, 0, sched_ints(c->n) * 4, s) != cudaSuccess) return MOE_ERR_CUDA;
    }
    const size_t R = static_cast<size_t>(c->k) * T;
    cudaError_t e = cudaSuccess;
    if (topk_idx && R) e = cudaMemcpyAsync(topk_idx, c->topk_idx, R * 4, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess && topk_w && R) e = cudaMemcpyAsync(topk_w, c->topk_w, R * 4, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess && counts) e = cudaMemcpyAsync(counts, c->sched, c->n * 4, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess && offsets)
        e = cudaMemcpyAsync(offsets, c->sched + c->n, (c->n + 1) * 4, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess && perm && R) e = cudaMemcpyAsync(perm, c->perm, R * 4, cudaMemcpyDeviceToDevice, s);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_router_logits(moe_ctx* c, const void* x, const float* Wg, int T, float* logits, moe_stream_t stream) {
    if (!c || T < 0) return MOE_ERR_INVALID;
    if (T == 0) return MOE_OK;
    if (!x || !Wg || !logits || !aligned16(x) || !aligned16(Wg)) return MOE_ERR_INVALID;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int rc = ensure_workspace(c, T, s);
    if (rc != MOE_OK) return rc;
    return run_route(c, x, Wg, T, s, logits, false);
}

int moe_forward(moe_ctx* c, const void* x, const float* Wg, const void* W1, const void* W3, const void* W2, void* y,
                int T, moe_stream_t stream) {
    if (!c || T < 0) return MOE_ERR_INVALID;
    if (T == 0) return MOE_OK;
    if (!x || !Wg || !W1 || !W3 || !W2 || !y) return MOE_ERR_INVALID;
    if (!aligned16(x) || !aligned16(Wg) || !aligned16(W1) || !aligned16(W3) || !aligned16(W2) || !aligned16(y))
        return MOE_ERR_INVALID;
    if (c->dtype == MOE_BF16 && !tc_shape_ok(c)) return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int rc = ensure_workspace(c, T, s, use_decode(c, T));
    if (rc != MOE_OK) return rc;
    return run_forward(c, x, Wg, W1, W3, W2, y, T, s);
}

int moe_block_forward(moe_ctx* c, void* h, float eps, const float* Wg, const void* W1, const void* W3,
                      const void* W2, int T, moe_stream_t stream) {
    if (!c || T < 0 || !(eps >= 0.0f)) return MOE_ERR_INVALID;
    if (T == 0) return MOE_OK;
    if (!h || !Wg || !W1 || !W3 || !W2) return MOE_ERR_INVALID;
    if (!aligned16(h) || !aligned16(Wg) || !aligned16(W1) || !aligned16(W3) || !aligned16(W2)) return MOE_ERR_INVALID;
    if (c->dtype == MOE_BF16 && !tc_shape_ok(c)) return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int rc = ensure_workspace(c, T, s, use_decode(c, T));
    if (rc != MOE_OK) return rc;
    return run_forward(c, h, Wg, W1, W3, W2, h, T, s, eps, h);
}

int moe_stack_forward(moe_ctx* c, void* h, float eps, int n_layers, const float* const* Wg, const void* const* W1,
                      const void* const* W3, const void* const* W2, int T, moe_stream_t stream) {
    if (!c || T < 0 || n_layers < 0 || !(eps >= 0.0f)) return MOE_ERR_INVALID;
    if (T == 0 || n_layers == 0) return MOE_OK;
    if (!h || !Wg || !W1 || !W3 || !W2) return MOE_ERR_INVALID;
    for (int l = 0; l < n_layers; ++l) {
        if (!Wg[l] || !W1[l] || !W3[l] || !W2[l]) return MOE_ERR_INVALID;
        if (!aligned16(Wg[l]) || !aligned16(W1[l]) || !aligned16(W3[l]) || !aligned16(W2[l])) return MOE_ERR_INVALID;
    }
    if (!aligned16(h)) return MOE_ERR_INVALID;
    if (c->dtype == MOE_BF16 && !tc_shape_ok(c)) return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int rc = ensure_workspace(c, T, s, use_decode(c, T));
    if (rc != MOE_OK) return rc;
    for (int l = 0; l < n_layers && rc == MOE_OK; ++l) rc = run_forward(c, h, Wg[l], W1[l], W3[l], W2[l], h, T, s, eps, h);
    return rc;
}

int moe_forward_fp8(moe_ctx* c, const void* x, const float* Wg, const uint8_t* W1q, const float* W1s,
                    const uint8_t* W3q, const float* W3s, const uint8_t* W2q, const float* W2s, void* y, int T,
                    moe_stream_t stream) {
    if (!c || T < 0) return MOE_ERR_INVALID;
    if (T == 0) return MOE_OK;
    if (!x || !Wg || !W1q || !W1s || !W3q || !W3s || !W2q || !W2s || !y) return MOE_ERR_INVALID;
    if (!aligned16(x) || !aligned16(Wg) || !aligned16(W1q) || !aligned16(W3q) || !aligned16(W2q) || !aligned16(y))
        return MOE_ERR_INVALID;
    auto aligned4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
    if (!aligned4(W1s) || !aligned4(W3s) || !aligned4(W2s)) return MOE_ERR_INVALID;
    if (c->dtype != MOE_BF16 || !tc_shape_ok(c) || c->n > 31) return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int chunk = T < kDecodeMaxT ? T : kDecodeMaxT;
    int rc = ensure_workspace(c, chunk, s, true);
    if (rc != MOE_OK) return rc;
    const size_t row_bytes = static_cast<size_t>(c->d) * 2;
    for (int t0 = 0; t0 < T && rc == MOE_OK; t0 += chunk) {
        const int Tc = T - t0 < chunk ? T - t0 : chunk;
        rc = run_forward_fp8(c, static_cast<const char*>(x) + t0 * row_bytes, Wg, W1q, W1s, W3q, W3s, W2q, W2s,
                             static_cast<char*>(y) + t0 * row_bytes, Tc, s);
    }
    return rc;
}

int moe_forward_host(moe_ctx* c, const void* x_host, const float* Wg, const void* W1, const void* W3, const void* W2,
                     void* y_host, int T, moe_stream_t stream) {
    if (!c || T < 0) return MOE_ERR_INVALID;
    if (T == 0) return MOE_OK;
    if (!x_host || !y_host) return MOE_ERR_INVALID;
    if (!Wg || !W1 || !W3 || !W2) return MOE_ERR_INVALID;
    if (c->dtype == MOE_BF16 && !tc_shape_ok(c)) return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int rc = ensure_workspace(c, T, s, use_decode(c, T));
    if (rc != MOE_OK) return rc;
    const size_t bytes = static_cast<size_t>(T) * c->d * esize(c->dtype);
    // The input copy runs on the context's own stream into one of two staging
    // buffers, so it can overlap the previous call's kernels; the layer and the
    // output copy stay on `stream`.  Reusing a staging buffer waits for the call
    // that read it.  While `stream` is being captured, everything stays on it.
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const bool capturing = cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone;
    void* xb = c->xbuf;
    if (!capturing && ensure_copy_stream(c)) {
        const int b = c->host_slot;
        c->host_slot ^= 1;
        xb = b ? c->xbuf2 : c->xbuf;
        if (cudaStreamWaitEvent(c->h2d_stream, c->ev_xfree[b], 0) != cudaSuccess ||
            cudaMemcpyAsync(xb, x_host, bytes, cudaMemcpyHostToDevice, c->h2d_stream) != cudaSuccess ||
            cudaEventRecord(c->ev_h2d[b], c->h2d_stream) != cudaSuccess || cudaStreamWaitEvent(s, c->ev_h2d[b], 0) != cudaSuccess)
            return MOE_ERR_CUDA;
        void* y_direct = c->host_out ? mapped_host_alias(y_host) : nullptr;
        rc = run_forward(c, xb, Wg, W1, W3, W2, y_direct ? y_direct : c->ybuf, T, s);
        if (rc != MOE_OK) return rc;
        if (cudaEventRecord(c->ev_xfree[b], s) != cudaSuccess) return MOE_ERR_CUDA;
        if (y_direct) return MOE_OK;   // the kernels wrote y into host memory
    } else {
        cudaGetLastError();
        if (cudaMemcpyAsync(xb, x_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) return MOE_ERR_CUDA;
        rc = run_forward(c, xb, Wg, W1, W3, W2, c->ybuf, T, s);
        if (rc != MOE_OK) return rc;
    }
    if (cudaMemcpyAsync(y_host, c->ybuf, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

int moe_status(moe_ctx* c) {
    if (!c) return MOE_ERR_INVALID;
    const int w = *reinterpret_cast<volatile int*>(c->status_host);
    if (w & kStatusTimeout) return MOE_ERR_TIMEOUT;
    if (w & kStatusBounds) return MOE_ERR_BOUNDS;
    return MOE_OK;
}

int moe_clear_status(moe_ctx* c) {
    if (!c) return MOE_ERR_INVALID;
    // A call that gave up (a bounded wait ran out) can leave the routing
    // kernel's barrier words or the fused combine's counters mid-count: put
    // them back (synchronously, on the device of the context).
    if (c->xchg && (*reinterpret_cast<volatile int*>(c->status_host) & kStatusTimeout)) {
        if (cudaDeviceSynchronize() != cudaSuccess ||
            cudaMemset(c->xchg, 0, static_cast<size_t>(reinterpret_cast<char*>(c->rstd) - reinterpret_cast<char*>(c->xchg))) !=
                cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
    }
    *reinterpret_cast<volatile int*>(c->status_host) = 0;
    return MOE_OK;
}

int moe_selftest_wait_timeout(moe_ctx* c, long long wait_limit_us, moe_stream_t stream) {
    if (!c || wait_limit_us <= 0 || wait_limit_us > 10000000) return MOE_ERR_INVALID;
    KStatus st = kstatus(c);
    st.wait_ns = static_cast<uint64_t>(wait_limit_us) * 1000ull;
    cudaError_t e = launch_wait_selftest(st, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_stage_times(moe_ctx* c, float* ms, int max_stages, int* calls) {
    if (!c || (max_stages > 0 && !ms)) return MOE_ERR_INVALID;
    const int ncalls = static_cast<int>(c->ev_calls.size());
    if (calls) *calls = ncalls;
    double sum[kStages] = {0};
    int rc = kStages;
    if (ncalls > 0) {
        if (cudaEventSynchronize(c->ev_calls.back()[kStages]) != cudaSuccess) rc = MOE_ERR_CUDA;
        for (auto& ev : c->ev_calls) {
            for (int i = 0; i < kStages && rc >= 0; ++i) {
                float t = 0.0f;
                if (cudaEventElapsedTime(&t, ev[i], ev[i + 1]) != cudaSuccess) rc = MOE_ERR_CUDA;
                sum[i] += t;
            }
            for (int i = 0; i <= kStages; ++i) c->ev_free.push_back(ev[i]);
        }
        c->ev_calls.clear();
    }
    if (rc < 0) {
        cudaGetLastError();
        return rc;
    }
    for (int i = 0; i < kStages && i < max_stages; ++i) ms[i] = ncalls ? static_cast<float>(sum[i] / ncalls) : 0.0f;
    return kStages;
}

const char* moe_stage_name(int i) { return (i >= 0 && i < kStages) ? kStageNames[i] : nullptr; }

const char* moe_error_string(int code) {
    switch (code) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID: return "MOE_ERR_INVALID";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_OOM: return "MOE_ERR_OOM";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_BOUNDS: return "MOE_ERR_BOUNDS";
        case MOE_ERR_SCRATCH_LIMIT: return "MOE_ERR_SCRATCH_LIMIT";
        default: return "MOE_ERR_UNKNOWN";
    }
}

void moe_destroy(moe_ctx* c) {
    if (!c) return;
    for (auto& ev : c->ev_calls) c->ev_free.insert(c->ev_free.end(), ev.begin(), ev.begin() + kStages + 1);
    for (cudaEvent_t e : c->ev_free) cudaEventDestroy(e);
    if (c->h2d_stream) {
        cudaStreamSynchronize(c->h2d_stream);
        cudaStreamDestroy(c->h2d_stream);
    }
    for (int i = 0; i < 2; ++i) {
        if (c->ev_h2d[i]) cudaEventDestroy(c->ev_h2d[i]);
        if (c->ev_xfree[i]) cudaEventDestroy(c->ev_xfree[i]);
    }
    if (c->ws) cudaFree(c->ws);
    if (c->status_host) cudaFreeHost(c->status_host);
    delete c;
}

}  // extern "C"
