// QK-norm + RoPE + KV append, and split-KV grouped-query decode attention
// over the static per-row cache [maxB][nkv][cap][128].
//
// The method: per-head RMSNorm of q and of k, each with its own weight
// (q and k normalised separately, Mizuoto "Qwen3-TTS" page, section "速度"),
// rotate-half RoPE at the absolute position with inv_freq held in fp32
// (same page, section "对照结果"), GQA where q head h reads kv head
// h / (nq/nkv) (repeat_interleave over heads, ncnn discussion 6798,
// section 2), causal softmax over positions 0..pos.
#include "common.cuh"
#include "kernels.h"

namespace q3 {

// ------------------------------------------------------------------ QK-norm, RoPE, KV append
// grid: M tokens; block: 32 * (nq + nkv) threads.  Warp w < nq: q head w;
// otherwise k head w - nq (and the matching v head is copied to the cache).
// Lane l holds head elements l, l+32, l+64, l+96: the RoPE pairs (j, j+64)
// for j = l and j = l+32 stay inside the lane.
template <typename T>
__global__ void qk_rope_kv_kernel(float* __restrict__ qkv, int ldq, int nq, int nkv, const float* __restrict__ qn,
                                  const float* __restrict__ kn, float eps, const float2* __restrict__ rope,
                                  int rope_rows, T* __restrict__ Kc, T* __restrict__ Vc, int cap,
                                  const int* __restrict__ tok_row, const int* __restrict__ tok_pos, int* err) {
    const int m = blockIdx.x;
    const int pos = tok_pos[m];
    if (pos < 0) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (pos >= cap || pos >= rope_rows) {
        if (threadIdx.x == 0) atomicOr(err, ERRB_BOUNDS);
        return;
    }
    const int row = tok_row[m];
    float* t = qkv + (size_t)m * ldq;
    const bool is_q = warp < nq;
    const int head = is_q ? warp : warp - nq;
    float* src = t + (size_t)(is_q ? head : nq + head) * HD;
    const float* wn = is_q ? qn : kn;
    float e[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) e[i] = src[lane + 32 * i];
    float ss = warp_sum(e[0] * e[0] + e[1] * e[1] + e[2] * e[2] + e[3] * e[3]);
    const float r = 1.0f / sqrtf(ss / (float)HD + eps);
#pragma unroll
    for (int i = 0; i < 4; ++i) e[i] = e[i] * r * wn[lane + 32 * i];
    const float2 cs0 = rope[(size_t)pos * (HD / 2) + lane];
    const float2 cs1 = rope[(size_t)pos * (HD / 2) + lane + 32];
    float a = e[0], b = e[2];
    e[0] = a * cs0.x - b * cs0.y;
    e[2] = b * cs0.x + a * cs0.y;
    a = e[1]; b = e[3];
    e[1] = a * cs1.x - b * cs1.y;
    e[3] = b * cs1.x + a * cs1.y;
    if (is_q) {
#pragma unroll
        for (int i = 0; i < 4; ++i) src[lane + 32 * i] = e[i];
    } else {
        const size_t off = (((size_t)row * nkv + head) * cap + pos) * HD;
        const float* v = t + (size_t)(nq + nkv + head) * HD;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            Kc[off + lane + 32 * i] = from_f<T>(e[i]);
            Vc[off + lane + 32 * i] = from_f<T>(v[lane + 32 * i]);
        }
    }
}

cudaError_t launch_qk_rope_kv(int dtype, float* qkv, int ldq, int M, int nq, int nkv, const float* q_norm,
                              const float* k_norm, float eps, const float* rope_cs, int rope_rows, void* Kc, void* Vc,
                              int cap, const int* tok_row, const int* tok_pos, int* err, cudaStream_t st) {
    if (M <= 0) return cudaSuccess;
    const int threads = 32 * (nq + nkv);
    if (dtype == Q3_BF16)
        qk_rope_kv_kernel<bf16><<<M, threads, 0, st>>>(qkv, ldq, nq, nkv, q_norm, k_norm, eps, (const float2*)rope_cs,
                                                       rope_rows, (bf16*)Kc, (bf16*)Vc, cap, tok_row, tok_pos, err);
    else
        qk_rope_kv_kernel<float><<<M, threads, 0, st>>>(qkv, ldq, nq, nkv, q_norm, k_norm, eps,
                                                        (const float2*)rope_cs, rope_rows, (float*)Kc, (float*)Vc, cap,
                                                        tok_row, tok_pos, err);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ split-KV attention
// grid (n_splits, nkv, M), 128 threads.  8 lanes cover one cached position
// (16 dims each), a warp walks 4 positions at a time, the block 16.  Each
// 8-lane group keeps an online softmax (running max, sum, weighted V) per q
// head of the kv group; groups then warps are merged, and the block writes
// its unnormalised partial for the split.
template <typename T, int GQ>
__global__ void __launch_bounds__(128) attn_split_kernel(const float* __restrict__ qkv, int ldq, int nq, int nkv,
                                                         const T* __restrict__ Kc, const T* __restrict__ Vc, int cap,
                                                         const int* __restrict__ tok_row,
                                                         const int* __restrict__ tok_pos, int n_splits,
                                                         float* __restrict__ pm, float* __restrict__ pl,
                                                         float* __restrict__ pacc) {
    const int split = blockIdx.x, g = blockIdx.y, m = blockIdx.z;
    const int pos = tok_pos[m];
    if (pos < 0) return;
    const int n = pos + 1;
    const int chunk = (n + n_splits - 1) / n_splits;
    const int j0 = split * chunk, j1 = min(n, j0 + chunk);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane & 7, grp = lane >> 3;
    const int d0 = sub * 16;
    const float scale = 0.08838834764831845f;  // 1/sqrt(128)

    float q[GQ][16];
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
        const float* qs = qkv + (size_t)m * ldq + (size_t)(g * GQ + hh) * HD + d0;
#pragma unroll
        for (int i = 0; i < 16; ++i) q[hh][i] = qs[i] * scale;
    }
    float mx[GQ], l[GQ], acc[GQ][16];
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
        mx[hh] = -INFINITY; l[hh] = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[hh][i] = 0.f;
    }
    const size_t base = ((size_t)tok_row[m] * nkv + g) * cap * HD;
    // the trip count is uniform over the warp (every lane runs the shuffles);
    // a group whose position is past the split's end only skips the update
    for (int jb = j0 + warp * 4; jb < j1; jb += 16) {
        const int j = jb + grp;
        const bool valid = j < j1;
        float k[16], v[16];
        if (valid) {
            float a[8], b[8];
            load8(Kc + base + (size_t)j * HD + d0, a);
            load8(Kc + base + (size_t)j * HD + d0 + 8, b);
#pragma unroll
            for (int i = 0; i < 8; ++i) { k[i] = a[i]; k[8 + i] = b[i]; }
            load8(Vc + base + (size_t)j * HD + d0, a);
            load8(Vc + base + (size_t)j * HD + d0 + 8, b);
#pragma unroll
            for (int i = 0; i < 8; ++i) { v[i] = a[i]; v[8 + i] = b[i]; }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) { k[i] = 0.f; v[i] = 0.f; }
        }
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) s = fmaf(q[hh][i], k[i], s);
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            s += __shfl_xor_sync(0xffffffffu, s, 4);
            if (valid) {
                const float mn = fmaxf(mx[hh], s);
                const float c = expf(mx[hh] - mn);
                const float p = expf(s - mn);
                l[hh] = l[hh] * c + p;
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[hh][i] = fmaf(p, v[i], acc[hh][i] * c);
                mx[hh] = mn;
            }
        }
    }
    // merge the 4 position groups of the warp (lanes sub, sub+8, sub+16, sub+24)
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
        float ma = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 8));
        ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 16));
        const float c = (ma == -INFINITY) ? 0.f : expf(mx[hh] - ma);
        float lv = l[hh] * c;
        lv += __shfl_xor_sync(0xffffffffu, lv, 8);
        lv += __shfl_xor_sync(0xffffffffu, lv, 16);
        l[hh] = lv;
        mx[hh] = ma;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float a = acc[hh][i] * c;
            a += __shfl_xor_sync(0xffffffffu, a, 8);
            a += __shfl_xor_sync(0xffffffffu, a, 16);
            acc[hh][i] = a;
        }
    }
    __shared__ float s_m[4][GQ], s_l[4][GQ], s_acc[4][GQ][HD];
    if (grp == 0) {
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
#pragma unroll
            for (int i = 0; i < 16; ++i) s_acc[warp][hh][d0 + i] = acc[hh][i];
            if (sub == 0) { s_m[warp][hh] = mx[hh]; s_l[warp][hh] = l[hh]; }
        }
    }
    __syncthreads();
    const int t = threadIdx.x;  // one head dimension per thread
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
        float ma = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) ma = fmaxf(ma, s_m[w][hh]);
        float lsum = 0.f, a = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float c = (ma == -INFINITY) ? 0.f : expf(s_m[w][hh] - ma);
            lsum += s_l[w][hh] * c;
            a += s_acc[w][hh][t] * c;
        }
        const size_t pi = ((size_t)m * n_splits + split) * nq + g * GQ + hh;
        pacc[pi * HD + t] = a;
        if (t == 0) { pm[pi] = ma; pl[pi] = lsum; }
    }
}

// grid (M, nq), 128 threads (one head dimension each): merge the splits of
// one head into the O-projection input; skipped tokens get zeros.
__global__ void __launch_bounds__(128) attn_combine_kernel(const float* __restrict__ pm, const float* __restrict__ pl,
                                                           const float* __restrict__ pacc, int n_splits, int nq,
                                                           const int* __restrict__ tok_pos, float* __restrict__ out,
                                                           int ldo, bf16* __restrict__ hi, bf16* __restrict__ lo) {
    const int m = blockIdx.x, h = blockIdx.y, t = threadIdx.x;
    float res = 0.f;
    if (tok_pos[m] >= 0) {
        float ma = -INFINITY;
        for (int s = 0; s < n_splits; ++s) ma = fmaxf(ma, pm[((size_t)m * n_splits + s) * nq + h]);
        float den = 0.f, num = 0.f;
        for (int s = 0; s < n_splits; ++s) {
            const size_t pi = ((size_t)m * n_splits + s) * nq + h;
            const float c = (pm[pi] == -INFINITY) ? 0.f : expf(pm[pi] - ma);
            den += pl[pi] * c;
            num += pacc[pi * HD + t] * c;
        }
        res = num / den;
    }
    const size_t i = (size_t)h * HD + t;
    if (hi) {
        // the O projection's tensor-core operand: bf16 high and low parts, [M][nq * 128]
        const bf16 hv = __float2bfloat16_rn(res);
        hi[(size_t)m * nq * HD + i] = hv;
        lo[(size_t)m * nq * HD + i] = __float2bfloat16_rn(res - __bfloat162float(hv));
    } else {
        out[(size_t)m * ldo + i] = res;
    }
}

template <typename T>
static cudaError_t attention_impl(const float* qkv, int ldq, int M, int nq, int nkv, const T* Kc, const T* Vc, int cap,
                                  const int* tok_row, const int* tok_pos, int n_splits, float* pm, float* pl,
                                  float* pacc, float* out, int ldo, bf16* hi, bf16* lo, cudaStream_t st) {
    dim3 grid(n_splits, nkv, M);
    const int gq = nq / nkv;
    switch (gq) {
        case 1: attn_split_kernel<T, 1><<<grid, 128, 0, st>>>(qkv, ldq, nq, nkv, Kc, Vc, cap, tok_row, tok_pos, n_splits, pm, pl, pacc); break;
        case 2: attn_split_kernel<T, 2><<<grid, 128, 0, st>>>(qkv, ldq, nq, nkv, Kc, Vc, cap, tok_row, tok_pos, n_splits, pm, pl, pacc); break;
        case 4: attn_split_kernel<T, 4><<<grid, 128, 0, st>>>(qkv, ldq, nq, nkv, Kc, Vc, cap, tok_row, tok_pos, n_splits, pm, pl, pacc); break;
        default: return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    attn_combine_kernel<<<dim3(M, nq), 128, 0, st>>>(pm, pl, pacc, n_splits, nq, tok_pos, out, ldo, hi, lo);
    return cudaGetLastError();
}

cudaError_t launch_attention(int dtype, const float* qkv, int ldq, int M, int nq, int nkv, const void* Kc,
                             const void* Vc, int cap, const int* tok_row, const int* tok_pos, int n_splits,
                             float* part_m, float* part_l, float* part_acc, float* out, int ldo, cudaStream_t st,
                             const TcScratch* split) {
    if (M <= 0) return cudaSuccess;
    bf16* hi = nullptr;
    bf16* lo = nullptr;
    if (split) {
        if (!tc_fits(*split, M, nq * HD)) return cudaErrorInvalidValue;
        hi = (bf16*)split->base;
        lo = hi + (size_t)M * nq * HD;
    }
    if (dtype == Q3_BF16)
        return attention_impl<bf16>(qkv, ldq, M, nq, nkv, (const bf16*)Kc, (const bf16*)Vc, cap, tok_row, tok_pos,
                                    n_splits, part_m, part_l, part_acc, out, ldo, hi, lo, st);
    return attention_impl<float>(qkv, ldq, M, nq, nkv, (const float*)Kc, (const float*)Vc, cap, tok_row, tok_pos,
                                 n_splits, part_m, part_l, part_acc, out, ldo, hi, lo, st);
}

}  // namespace q3
