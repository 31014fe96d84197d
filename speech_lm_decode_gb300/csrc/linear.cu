// Projections of the talker / code predictor and the RMSNorm that feeds them.
// Weights are in the model dtype (bf16 or fp32); the input vectors (operands)
// and all accumulation are fp32.
//
// Small batches (M <= 8 rows) are weight-streaming GEMVs: a warp owns R output
// rows, lanes stream 16-byte chunks of the weight rows (read once, not kept
// in L1) and keep M running sums each; a fixed-order warp reduction follows.
// Larger M (prefill chunks, large batches) use the tensor-core path for bf16
// weights (gemm_tc.cu) and a shared-memory tiled CUDA-core GEMM otherwise.
#include "common.cuh"
#include "kernels.h"
#include "pdl.cuh"

namespace q3 {

// ------------------------------------------------------------------ GEMV
template <typename T, int M, int R, bool GATED>
__global__ void __launch_bounds__(128) gemv_kernel(const T* __restrict__ W, int N, int K,
                                                   const float* __restrict__ X, int ldx, float* __restrict__ Y,
                                                   int ldy, const float* __restrict__ bias, int accumulate, int F,
                                                   float* __restrict__ G, int ldg) {
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = (blockIdx.x * 4 + warp) * R;
    if (n0 >= N) return;
    float acc[R][M], accu[GATED ? R : 1][M];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) { acc[r][m] = 0.f; if (GATED) accu[GATED ? r : 0][m] = 0.f; }

    for (int k = lane * 8; k < K; k += 256) {
        float x[M][8];
#pragma unroll
        for (int m = 0; m < M; ++m) load8(X + (size_t)m * ldx + k, x[m]);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int n = min(n0 + r, N - 1);
            float w[8];
            load8_stream(W + (size_t)n * K + k, w);
#pragma unroll
            for (int m = 0; m < M; ++m)
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[r][m] = fmaf(w[i], x[m][i], acc[r][m]);
            if (GATED) {
                float u[8];
                load8_stream(W + (size_t)(F + n) * K + k, u);
#pragma unroll
                for (int m = 0; m < M; ++m)
#pragma unroll
                    for (int i = 0; i < 8; ++i) accu[GATED ? r : 0][m] = fmaf(u[i], x[m][i], accu[GATED ? r : 0][m]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int n = n0 + r;
#pragma unroll
        for (int m = 0; m < M; ++m) {
            float v = warp_sum(acc[r][m]);
            float u = GATED ? warp_sum(accu[GATED ? r : 0][m]) : 0.f;
            if (lane == 0 && n < N) {
                if (GATED) {
                    G[(size_t)m * ldg + n] = v / (1.0f + expf(-v)) * u;
                } else {
                    if (bias) v += bias[n];
                    float* y = Y + (size_t)m * ldy + n;
                    *y = accumulate ? *y + v : v;
                }
            }
        }
    }
}

// ------------------------------------------------------------------ tiled GEMM
constexpr int TBM = 64, TBN = 64, TBK = 16;

template <typename T, bool GATED>
__global__ void __launch_bounds__(256) gemm_tiled(const T* __restrict__ W, int N, int K,
                                                  const float* __restrict__ X, int ldx, int M,
                                                  float* __restrict__ Y, int ldy, const float* __restrict__ bias,
                                                  int accumulate, int F, float* __restrict__ G, int ldg) {
    pdl_wait();
    pdl_trigger();
    __shared__ float xs[TBK][TBM + 4];
    __shared__ float ws[TBK][TBN + 4];
    __shared__ float us[GATED ? TBK : 1][TBN + 4];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int m0 = blockIdx.y * TBM, n0 = blockIdx.x * TBN;
    float acc[4][4] = {}, accu[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += TBK) {
        for (int e = threadIdx.x; e < TBM * TBK; e += 256) {
            const int r = e / TBK, c = e % TBK;
            const int m = m0 + r, n = n0 + r, k = k0 + c;
            xs[c][r] = (m < M && k < K) ? X[(size_t)m * ldx + k] : 0.f;
            ws[c][r] = (n < N && k < K) ? to_f(W[(size_t)n * K + k]) : 0.f;
            if (GATED) us[GATED ? c : 0][r] = (n < N && k < K) ? to_f(W[(size_t)(F + n) * K + k]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int c = 0; c < TBK; ++c) {
            float a[4], b[4], bu[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) { a[i] = xs[c][ty * 4 + i]; b[i] = ws[c][tx * 4 + i]; }
            if (GATED) {
#pragma unroll
                for (int i = 0; i < 4; ++i) bu[i] = us[GATED ? c : 0][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
                    if (GATED) accu[i][j] = fmaf(a[i], bu[j], accu[i][j]);
                }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= N) continue;
            float v = acc[i][j];
            if (GATED) {
                G[(size_t)m * ldg + n] = v / (1.0f + expf(-v)) * accu[i][j];
            } else {
                if (bias) v += bias[n];
                float* y = Y + (size_t)m * ldy + n;
                *y = accumulate ? *y + v : v;
            }
        }
    }
}

template <typename T, bool GATED>
static cudaError_t linear_impl(const T* W, int N, int K, const float* X, int ldx, int M, float* Y, int ldy,
                               const float* bias, int accumulate, int F, float* G, int ldg, cudaStream_t st) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    if (M <= 8) {
        // rows per warp: 2 when there are enough rows to cover the GPU twice over
        const bool two = (N >= 4 * 2 * device_sm_count() * 2);
        const int rows_per_block = 4 * (two ? 2 : 1);
        dim3 grid((N + rows_per_block - 1) / rows_per_block);
#define GEMV_CASE(MM)                                                                                           \
    case MM:                                                                                                     \
        if (two) launch_pdl(gemv_kernel<T, MM, 2, GATED>, grid, 128, 0, st, W, N, K, X, ldx, Y, ldy, bias, accumulate, F, G, ldg); \
        else launch_pdl(gemv_kernel<T, MM, 1, GATED>, grid, 128, 0, st, W, N, K, X, ldx, Y, ldy, bias, accumulate, F, G, ldg);     \
        break;
        switch (M) {
            GEMV_CASE(1) GEMV_CASE(2) GEMV_CASE(3) GEMV_CASE(4) GEMV_CASE(5) GEMV_CASE(6) GEMV_CASE(7) GEMV_CASE(8)
        }
#undef GEMV_CASE
    } else {
        dim3 grid((N + TBN - 1) / TBN, (M + TBM - 1) / TBM);
        launch_pdl(gemm_tiled<T, GATED>, grid, 256, 0, st, W, N, K, X, ldx, M, Y, ldy, bias, accumulate, F, G, ldg);
    }
    return cudaGetLastError();
}

int device_sm_count() {
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    if (!cache[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 1;
    }
    return cache[dev];
}

static bool use_tc(int dtype, int M, const TcScratch& tc) {
    return dtype == Q3_BF16 && tc.min_tokens > 0 && M >= tc.min_tokens && tc_available();
}

bool linear_takes_split(int dtype, int M, int K, const TcScratch& tc) { return use_tc(dtype, M, tc) && tc_fits(tc, M, K); }

cudaError_t launch_linear(int dtype, const void* W, int N, int K, const float* X, int ldx, int M, float* Y, int ldy,
                          const float* bias, int accumulate, const TcScratch& tc, int* err, cudaStream_t st) {
    if (linear_takes_split(dtype, M, K, tc))
        return launch_linear_tc(W, N, K, X, ldx, M, Y, ldy, bias, accumulate, tc, err, st);
    if (!X) return cudaErrorInvalidValue;
    if (dtype == Q3_BF16)
        return linear_impl<bf16, false>((const bf16*)W, N, K, X, ldx, M, Y, ldy, bias, accumulate, 0, nullptr, 0, st);
    return linear_impl<float, false>((const float*)W, N, K, X, ldx, M, Y, ldy, bias, accumulate, 0, nullptr, 0, st);
}

cudaError_t launch_linear_gated(int dtype, const void* W, int F, int K, const float* X, int ldx, int M, float* out,
                                int ldo, const TcScratch& tc, int* err, cudaStream_t st, const TcScratch* out_split) {
    if (linear_takes_split(dtype, M, K, tc))
        return launch_linear_gated_tc(W, F, K, X, ldx, M, out, ldo, tc, err, st, out_split);
    if (!X || out_split) return cudaErrorInvalidValue;
    if (dtype == Q3_BF16)
        return linear_impl<bf16, true>((const bf16*)W, F, K, X, ldx, M, nullptr, 0, nullptr, 0, F, out, ldo, st);
    return linear_impl<float, true>((const float*)W, F, K, X, ldx, M, nullptr, 0, nullptr, 0, F, out, ldo, st);
}

// ------------------------------------------------------------------ RMSNorm
// hi != NULL: the output goes to hi / lo (bf16 parts, row stride n) instead of out
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* __restrict__ x, int ldx, const float* __restrict__ w,
                                                      int n, float eps, float* __restrict__ out, int ldo,
                                                      float* __restrict__ hout, int ldh, const int* __restrict__ out_row,
                                                      bf16* __restrict__ hi, bf16* __restrict__ lo) {
    pdl_wait();
    pdl_trigger();
    const int m = blockIdx.x;
    const int orow = out_row ? out_row[m] : m;
    if (orow < 0) return;
    const float* xr = x + (size_t)m * ldx;
    float ss = 0.f;
    for (int i = threadIdx.x; i < n; i += 256) ss = fmaf(xr[i], xr[i], ss);
    __shared__ float red[8];
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < 8 ? red[threadIdx.x] : 0.f;
        v = warp_sum(v);
        if (threadIdx.x == 0) red[0] = v;
    }
    __syncthreads();
    const float r = 1.0f / sqrtf(red[0] / (float)n + eps);
    for (int i = threadIdx.x; i < n; i += 256) {
        const float y = xr[i] * r * w[i];
        if (hi) {
            const bf16 h = __float2bfloat16_rn(y);
            hi[(size_t)orow * n + i] = h;
            lo[(size_t)orow * n + i] = __float2bfloat16_rn(y - __bfloat162float(h));
        } else {
            out[(size_t)orow * ldo + i] = y;
        }
        if (hout) hout[(size_t)orow * ldh + i] = y;
    }
}

cudaError_t launch_rmsnorm(const float* x, int ldx, int M, const float* w, int n, float eps, float* out, int ldo,
                           float* hout, int ldh, const int* out_row, cudaStream_t st) {
    if (M <= 0) return cudaSuccess;
    launch_pdl(rmsnorm_kernel, M, 256, 0, st, x, ldx, w, n, eps, out, ldo, hout, ldh, out_row, nullptr, nullptr);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm_split(const float* x, int ldx, int M, const float* w, int n, float eps,
                                 const TcScratch& tc, cudaStream_t st) {
    if (M <= 0) return cudaSuccess;
    if (!tc_fits(tc, M, n)) return cudaErrorInvalidValue;
    bf16* hi = (bf16*)tc.base;
    launch_pdl(rmsnorm_kernel, M, 256, 0, st, x, ldx, w, n, eps, nullptr, 0, nullptr, 0, nullptr, hi, hi + (size_t)M * n);
    return cudaGetLastError();
}

}  // namespace q3
