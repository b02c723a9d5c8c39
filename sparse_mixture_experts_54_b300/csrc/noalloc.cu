// noalloc.cu -- moe_forward_noalloc: the layer's forward call without any
// device or host allocation, for callers that cannot call cudaMalloc.
//
// Who needs it: code whose device memory is owned and budgeted by someone
// else (a serving process that hands the whole GPU to its own caching
// allocator, or one that must not allocate once it starts answering requests
// so that its memory footprint is fixed), and code that runs where an
// allocation would be unsafe or unwelcome (for example between the steps of
// a latency-critical loop, where cudaMalloc/cudaFree synchronise the device).
//
// Instead of the context's growable workspace, the scratch of the call --
// routing indices and gates, dispatch order and schedule, the gathered token
// rows, the SwiGLU rows and the per-slot expert outputs -- lives in one
// file-scope __device__ array of fixed size.  The CUDA module that holds it is
// loaded once per device, so every GPU that loads this library keeps the
// array until the process exits.  It launches the library's separate router,
// dispatch, gather, grouped-GEMM and combine kernels (moe_forward fuses some
// of these steps with the help of counters kept in its context's workspace),
// so its results agree with moe_forward's within the tests' tolerance.
#include <mutex>

#include "../../include/moe.h"
#include "kernels.h"

using namespace moe;

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;   // 32 MiB, the most one call may use
__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_dev[kMaxDevices];   // device address of g_noalloc_scratch, per device
int g_num_sms[kMaxDevices];

size_t up256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Once per device, with that device current: the array's device address.
// In host code the symbol names a host-side stand-in, never the device copy.
int scratch_for_device(int dev, unsigned char** ptr, int* sms) {
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_dev[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 148;
        }
        g_num_sms[dev] = n;
        g_scratch_dev[dev] = p;
    }
    *ptr = static_cast<unsigned char*>(g_scratch_dev[dev]);
    *sms = g_num_sms[dev];
    return MOE_OK;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int moe_forward_noalloc(const void* x, const float* W_g, const float* b_g, const void* W1,
                                   const void* W3, const void* W2, void* y, int T, int d, int d_ff, int n_experts,
                                   int k, int dtype, int* status, moe_stream_t stream) {
    if (T < 0 || d <= 0 || d % 8 != 0 || d_ff <= 0 || n_experts < 1 || n_experts > 32 || k < 1 || k > n_experts)
        return MOE_ERR_INVALID;
    if (dtype != MOE_BF16 && dtype != MOE_F32) return MOE_ERR_INVALID;
    if (static_cast<size_t>(n_experts) * d * 4 > 200 * 1024) return MOE_ERR_UNSUPPORTED;
    if (dtype == MOE_BF16 && (d % 256 != 0 || d_ff % 128 != 0)) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!x || !W_g || !W1 || !W3 || !W2 || !y) return MOE_ERR_INVALID;
    if (!al16(x) || !al16(W_g) || !al16(W1) || !al16(W3) || !al16(W2) || !al16(y) || (b_g && !al16(b_g)))
        return MOE_ERR_INVALID;

    // Scratch layout for this call; refuse anything beyond the fixed array.
    const size_t R = static_cast<size_t>(k) * static_cast<size_t>(T);
    const size_t es = dtype == MOE_F32 ? 4 : 2;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off += up256(bytes); return o; };
    const size_t o_idx = take(R * 4), o_w = take(R * 4), o_perm = take(R * 4), o_inv = take(R * 4);
    const size_t o_sched = take(static_cast<size_t>(sched_ints(n_experts)) * 4);
    const size_t o_xp = take(R * d * es), o_h = take(R * d_ff * es), o_ys = take(R * d * 4);
    if (off > kScratchBytes) return MOE_ERR_SCRATCH_LIMIT;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    unsigned char* base = nullptr;
    int sms = 148;
    int rc = scratch_for_device(dev, &base, &sms);
    if (rc != MOE_OK) return rc;

    int32_t* topk_idx = reinterpret_cast<int32_t*>(base + o_idx);
    float* topk_w = reinterpret_cast<float*>(base + o_w);
    int32_t* perm = reinterpret_cast<int32_t*>(base + o_perm);
    int32_t* inv = reinterpret_cast<int32_t*>(base + o_inv);
    int* sched = reinterpret_cast<int*>(base + o_sched);
    void* Xp = base + o_xp;
    void* H = base + o_h;
    float* Ys = reinterpret_cast<float*>(base + o_ys);

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    KStatus st;
    st.word = status;
    st.wait_ns = 2000000000ull;
    const ElemType et = dtype == MOE_F32 ? ElemType::F32 : ElemType::BF16;
    const int Ri = static_cast<int>(R);
    // Every scratch region below is fully written before it is read within
    // this call, so nothing depends on what an earlier call left behind.
    cudaError_t e = launch_router(et, x, W_g, b_g, T, d, n_experts, k, topk_idx, topk_w, nullptr, sms, s);
    if (e == cudaSuccess) e = launch_dispatch(topk_idx, Ri, n_experts, sched, perm, inv, st, s);
    if (e == cudaSuccess) e = launch_gather(et, x, perm, Ri, k, d, Xp, s);
    if (e == cudaSuccess) {
        if (et == ElemType::F32) {
            e = launch_simt_gemm13(et, Xp, W1, W3, H, sched, n_experts, d, d_ff, Ri, s);
            if (e == cudaSuccess)
                e = launch_simt_gemm2(et, H, W2, Ys, sched, perm, topk_w, n_experts, d, d_ff, Ri, s);
        } else {
            CUtensorMap mXp, mH, mW1, mW3, mW2;
            const uint64_t nF = static_cast<uint64_t>(n_experts) * d_ff, nd = static_cast<uint64_t>(n_experts) * d;
            if (!encode_map_bf16_2d(&mXp, Xp, R, d, 128) || !encode_map_bf16_2d(&mH, H, R, d_ff, 128) ||
                !encode_map_bf16_2d(&mW1, W1, nF, d, 128) || !encode_map_bf16_2d(&mW3, W3, nF, d, 128) ||
                !encode_map_bf16_2d(&mW2, W2, nd, d_ff, 256))
                return MOE_ERR_CUDA;
            e = launch_tc_gemm13(mXp, mW1, mW3, sched, n_experts, d, d_ff, Ri, static_cast<__nv_bfloat16*>(H), st,
                                 sms, s);
            if (e == cudaSuccess)
                e = launch_tc_gemm2(mH, mW2, sched, n_experts, d, d_ff, Ri, Ys, perm, topk_w, CombineArgs{}, st,
                                    sms, s);
        }
    }
    if (e == cudaSuccess) e = launch_combine(et, Ys, T, k, d, nullptr, y, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}
