// Calibration of the tensor-core GEMM's shape choice: CUDA-event time of every
// legal tile width (NT 32 / 64 / 128) and K split (1 / 2 / 4 / 8) over the
// projection shapes of the frame loop and the prefill (0.6B and 1.7B widths,
// 16..8192 tokens), with the operand already split and L2 flushed between
// repetitions (median of 10 after 2 warm-up launches).  Built by
// build.build_calibration() with Q3_GEMM_CALIBRATION; prints CSV.  The cost
// model in gemm_tc.cu (best_split) was fitted to this table.
#include <cstdio>
#include <vector>
#include <algorithm>
#include <cuda_runtime.h>
#include "kernels.h"
namespace q3 { extern int g_force_nt, g_force_ks; bool tc_shape_ok(int NT, int ks, bool gated, int K); }
using namespace q3;
#define CKE(x) do { cudaError_t e = (x); if (e != cudaSuccess) { printf("ERR %s line %d: %s\n", #x, __LINE__, cudaGetErrorString(e)); return 1; } } while (0)
int main() {
    struct S { const char* name; int N, K, gated; };
    std::vector<S> shapes = {{"qkv06", 4096, 1024, 0}, {"o06", 1024, 2048, 0}, {"gu06", 3072, 1024, 1}, {"d06", 1024, 3072, 0},
                             {"head06", 3072, 1024, 0}, {"cphead", 2048, 1024, 0},
                             {"qkv17", 4096, 2048, 0}, {"o17", 2048, 2048, 0}, {"gu17", 6144, 2048, 1}, {"d17", 2048, 6144, 0},
                             {"proj17", 1024, 2048, 0}};
    std::vector<int> Ms = {16, 32, 64, 256, 512, 8192};
    size_t wmax = 0, xmax = 0, ymax = 0;
    for (auto& s : shapes) { wmax = std::max(wmax, (size_t)s.N * (s.gated ? 2 : 1) * s.K * 2); xmax = std::max(xmax, (size_t)8192 * s.K * 4); ymax = std::max(ymax, (size_t)8192 * s.N * 4); }
    void *W, *X, *Y, *flush; int* err;
    CKE(cudaMalloc(&W, wmax)); CKE(cudaMalloc(&X, xmax)); CKE(cudaMalloc(&Y, ymax)); CKE(cudaMalloc(&flush, 512u << 20)); CKE(cudaMalloc(&err, 16));
    CKE(cudaMemset(W, 0x3c, wmax)); CKE(cudaMemset(X, 0x3c, xmax)); CKE(cudaMemset(err, 0, 16));
    cudaStream_t st; CKE(cudaStreamCreate(&st));
    cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
    TcScratch tc; tc.base = X; tc.bytes = xmax; tc.min_tokens = 1;
    printf("shape,N,K,gated,M,NT,ks,us_median\n");
    for (auto& s : shapes)
        for (int M : Ms)
            for (int nt : {32, 64, 128}) {
                if (nt > 32 && nt > (M + 31) / 32 * 32) continue;
                for (int ks : {1, 2, 4, 8}) {
                    if (!tc_shape_ok(nt, ks, s.gated, s.K)) continue;
                    g_force_nt = nt; g_force_ks = ks;
                    std::vector<float> t;
                    for (int r = 0; r < 12; ++r) {
                        CKE(cudaMemsetAsync(flush, r, 512u << 20, st));
                        CKE(cudaEventRecord(e0, st));
                        cudaError_t e = s.gated ? launch_linear_gated_tc(W, s.N, s.K, nullptr, s.K, M, (float*)Y, s.N, tc, err, st)
                                                : launch_linear_tc(W, s.N, s.K, nullptr, s.K, M, (float*)Y, s.N, nullptr, 0, tc, err, st);
                        if (e != cudaSuccess) { printf("ERR launch %s M %d nt %d ks %d: %s\n", s.name, M, nt, ks, cudaGetErrorString(e)); return 1; }
                        CKE(cudaEventRecord(e1, st));
                        CKE(cudaStreamSynchronize(st));
                        float ms; cudaEventElapsedTime(&ms, e0, e1);
                        if (r >= 2) t.push_back(ms * 1000.f);
                    }
                    std::sort(t.begin(), t.end());
                    printf("%s,%d,%d,%d,%d,%d,%d,%.2f\n", s.name, s.N, s.K, s.gated, M, nt, ks, t[t.size() / 2]);
                    fflush(stdout);
                }
            }
    int h = 0; cudaMemcpy(&h, err, 4, cudaMemcpyDeviceToHost);
    printf("err word %d\n", h);
    return 0;
}
