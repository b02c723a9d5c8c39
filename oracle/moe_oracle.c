/*
 * moe_oracle.c -- plain, slow, fp64 CPU oracle for the Mixtral sparse MoE
 * feed-forward layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library (the CUDA path) links,
 * includes or calls this file; it shares no code, header, table or constant
 * with it.  Only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark use it.
 *
 * What it computes, per token, independently (the MoE layer "is applied
 * independently per token": Mixtral deep dive (aiqianji), section 2.1.1):
 *
 *   l      = x . W_g^T (+ b)              router linear, nn.Linear(d, n, bias=False)
 *                                          (aiqianji section 2.1.4; code step 3 of 3.1.1)
 *   S      = the K largest l_i, descending; equal logits -> lower index first
 *   g_s    = exp(l_s - l_max) / sum_{s' in S} exp(l_s' - l_max)
 *                                          G(x) = Softmax(TopK(x . W_g)), TopK sets the
 *                                          others to -inf (aiqianji 2.1.1; xyznot "Method")
 *   E_e(x) = W2_e ( SiLU(W1_e x) * (W3_e x) ),  SiLU(z) = z / (1 + e^-z)
 *                                          (aiqianji 3.2.4, code block D; SwiGLU expert)
 *   y      = sum over slots k of g_k E_{S_k}(x), summed in slot order
 *                                          (aiqianji 2.1.1, y = sum_i Softmax(Top2(x W_g))_i SwiGLU_i(x))
 *
 * Dispatch reference: counts_e, exclusive-scan offsets, and the stable order of
 * assignments (t, k) by (expert, t*K + k); the one_hot/permute/where walk of
 * aiqianji 3.1.2 and code blocks B/C lists, per expert, the same tokens.
 *
 * Inputs are taken exactly as stored (bf16 bit patterns or fp32) and widened
 * exactly to double; every sum is a plain left-to-right double loop, no BLAS.
 * Weight layouts follow nn.Linear ([out][in]): W_g [n][d] fp32, W1/W3 [n][F][d],
 * W2 [n][d][F], x [T][d], all row-major.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_BF16 = 0, ORACLE_F32 = 1 };

/* A bf16 value is the upper half of an IEEE binary32; widening is exact. */
static double widen_bf16(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void* base, int64_t i, int dtype) {
    if (dtype == ORACLE_BF16) return widen_bf16(((const uint16_t*)base)[i]);
    return (double)((const float*)base)[i];
}

/* Widen n stored elements starting at element index i0 into out[]. */
void oracle_widen(const void* base, int dtype, int64_t i0, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = load_elem(base, i0 + i, dtype);
}

/* Router logits l[t][e] = sum_j x[t][j] * W_g[e][j]  (+ b[e] when b != NULL). */
int oracle_router_logits(const void* x, int x_dtype, const float* Wg, const float* b,
                         int64_t T, int d, int n, double* logits) {
    if (!x || !Wg || !logits || T < 0 || d <= 0 || n <= 0) return -1;
    for (int64_t t = 0; t < T; ++t) {
        for (int e = 0; e < n; ++e) {
            double acc = 0.0;
            for (int j = 0; j < d; ++j)
                acc += load_elem(x, t * (int64_t)d + j, x_dtype) * (double)Wg[(int64_t)e * d + j];
            if (b) acc += (double)b[e];
            logits[t * n + e] = acc;
        }
    }
    return 0;
}

/*
 * Top-K selection and gate softmax for each token.
 * Selection: repeatedly take the largest remaining logit; a strictly larger
 * value is needed to displace an earlier (lower) index, so equal logits go to
 * the lower expert index, which also takes the earlier slot.
 * Gate: softmax over the kept logits only (the TopK operator sets the rest to
 * -inf, whose exponentials are exactly zero), shifted by the slot-0 maximum.
 */
int oracle_select_topk(const double* logits, int64_t T, int n, int K,
                       int32_t* idx, double* gate) {
    if (!logits || !idx || !gate || K < 1 || K > n || n > 1024) return -1;
    for (int64_t t = 0; t < T; ++t) {
        const double* l = logits + t * n;
        unsigned char taken[1024];
        memset(taken, 0, (size_t)n);
        for (int k = 0; k < K; ++k) {
            int best = -1;
            for (int e = 0; e < n; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;
            }
            taken[best] = 1;
            idx[t * K + k] = best;
        }
        double lmax = l[idx[t * K + 0]];
        double z = 0.0;
        for (int k = 0; k < K; ++k) z += exp(l[idx[t * K + k]] - lmax);
        for (int k = 0; k < K; ++k) gate[t * K + k] = exp(l[idx[t * K + k]] - lmax) / z;
    }
    return 0;
}

/*
 * Dispatch: counts[e] = number of assignments (t,k) with idx[t][k] == e;
 * offsets = exclusive scan of counts (offsets[n] = K*T); perm lists the flat
 * assignment numbers t*K+k grouped by expert, ascending within each expert.
 */
int oracle_dispatch(const int32_t* idx, int64_t T, int K, int n,
                    int64_t* counts, int64_t* offsets, int64_t* perm) {
    if (!idx || !counts || !offsets || !perm || K < 1 || n < 1) return -1;
    int64_t R = T * K;
    for (int e = 0; e < n; ++e) counts[e] = 0;
    for (int64_t a = 0; a < R; ++a) {
        if (idx[a] < 0 || idx[a] >= n) return -2;
        counts[idx[a]] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < n; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int64_t pos = 0;
    for (int e = 0; e < n; ++e)
        for (int64_t a = 0; a < R; ++a)
            if (idx[a] == e) perm[pos++] = a;
    return 0;
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * One SwiGLU expert on one token row xr[d] (already widened):
 *   a_f = sum_j W1[e][f][j] x_j,  b_f = sum_j W3[e][f][j] x_j,
 *   h_f = SiLU(a_f) * b_f,        out_i = sum_f W2[e][i][f] h_f.
 * h must hold F doubles of scratch.
 */
static void expert_swiglu(const double* xr, const void* W1, const void* W3, const void* W2,
                          int w_dtype, int d, int F, int e, double* h, double* out) {
    int64_t w13 = (int64_t)e * F * d;
    for (int f = 0; f < F; ++f) {
        double a = 0.0, b = 0.0;
        int64_t row = w13 + (int64_t)f * d;
        for (int j = 0; j < d; ++j) {
            a += load_elem(W1, row + j, w_dtype) * xr[j];
            b += load_elem(W3, row + j, w_dtype) * xr[j];
        }
        h[f] = silu(a) * b;
    }
    int64_t w2 = (int64_t)e * d * F;
    for (int i = 0; i < d; ++i) {
        double o = 0.0;
        int64_t row = w2 + (int64_t)i * F;
        for (int f = 0; f < F; ++f) o += load_elem(W2, row + f, w_dtype) * h[f];
        out[i] = o;
    }
}

/* One expert on given token rows, no gate: out[s][d] = E_e(x[toks[s]]). */
int oracle_expert_rows(const void* x, int x_dtype, const void* W1, const void* W3, const void* W2,
                       int w_dtype, int d, int F, int e, const int64_t* toks, int64_t ntok,
                       double* out, double* scratch /* (d + F) doubles */) {
    if (!x || !W1 || !W3 || !W2 || !out || !scratch) return -1;
    double* xr = scratch;
    double* h = scratch + d;
    for (int64_t s = 0; s < ntok; ++s) {
        for (int j = 0; j < d; ++j) xr[j] = load_elem(x, toks[s] * (int64_t)d + j, x_dtype);
        expert_swiglu(xr, W1, W3, W2, w_dtype, d, F, e, h, out + s * d);
    }
    return 0;
}

/*
 * Sparse MoE output for the listed tokens, given each token's selection idx[t][K]
 * and gates gate[t][K] (indexed by the token number, not the list position):
 *   y[s][:] = sum_{k=0}^{K-1} gate[t][k] * E_{idx[t][k]}(x[t]),  t = toks[s].
 * Tokens are spread over nthreads OpenMP threads; each token is computed by
 * one thread, start to finish.  Scratch is malloc-free: caller passes
 * nthreads * (2*d + F) doubles.
 */
int oracle_moe_tokens(const void* x, int x_dtype, const void* W1, const void* W3, const void* W2,
                      int w_dtype, int d, int F, int n, int K, const int32_t* idx, const double* gate,
                      const int64_t* toks, int64_t ntok, double* y, int nthreads, double* scratch) {
    if (!x || !W1 || !W3 || !W2 || !idx || !gate || !toks || !y || !scratch) return -1;
    if (nthreads < 1) nthreads = 1;
    int bad = 0;
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1) reduction(| : bad)
#endif
    for (int64_t s = 0; s < ntok; ++s) {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        double* xr = scratch + (int64_t)tid * (2 * d + F);
        double* o = xr + d;
        double* h = o + d;
        int64_t t = toks[s];
        for (int j = 0; j < d; ++j) xr[j] = load_elem(x, t * (int64_t)d + j, x_dtype);
        double* ys = y + s * d;
        for (int i = 0; i < d; ++i) ys[i] = 0.0;
        for (int k = 0; k < K; ++k) {
            int e = idx[t * K + k];
            if (e < 0 || e >= n) { bad |= 1; continue; }
            expert_swiglu(xr, W1, W3, W2, w_dtype, d, F, e, h, o);
            double g = gate[t * K + k];
            for (int i = 0; i < d; ++i) ys[i] += g * o[i];
        }
    }
    return bad ? -2 : 0;
}

/* Number of OpenMP threads the oracle would use by default (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
