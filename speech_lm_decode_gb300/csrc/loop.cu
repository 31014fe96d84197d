// Per-step bookkeeping and embedding gathers of the frame loop.
//
// Talker input of step k (ncnn discussion 6798, section 1, generation loop):
// codec_emb(code0) + sum_{q=1..15} table[q-1](code_q) + trailing text row
// k-1 (tts_pad once the row's text is used up), summed in that order in fp32.
// Finished rows are fed EOS (Mizuoto "Qwen3-TTS" page, "与上游一致的做法").
// Predictor tokens of frame f: [h, codec_emb(code0)] at positions 0, 1, then
// table[s-1](code_s) at position s+1 (ncnn discussion 6798, section 1).
#include "common.cuh"
#include "kernels.h"
#include "pdl.cuh"

#include <algorithm>

namespace q3 {

// Token lists of this step: talker token b at the row's position; predictor
// prefill tokens (b, 0), (b, 1); predictor step s token (b, s+1).  Finished
// rows get position -1 (skipped by the KV append and attention).
__global__ void prepare_step_kernel(RowState* rs, int B, int* t_row, int* t_pos, int* c_row, int* c_pos, int G1) {
    pdl_wait();
    pdl_trigger();
    for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < B; b += gridDim.x * blockDim.x) {
        const bool live = !rs[b].finished;
        t_row[b] = b;
        t_pos[b] = live ? rs[b].pos : -1;
        c_row[2 * b] = b; c_pos[2 * b] = live ? 0 : -1;
        c_row[2 * b + 1] = b; c_pos[2 * b + 1] = live ? 1 : -1;
        for (int s = 1; s < G1; ++s) {
            c_row[(size_t)s * 2 * B + b] = b;
            c_pos[(size_t)s * 2 * B + b] = live ? s + 1 : -1;
        }
    }
}

cudaError_t launch_prepare_step(RowState* rs, int B, int* t_row, int* t_pos, int* c_row, int* c_pos, int G1,
                                cudaStream_t st) {
    launch_pdl(prepare_step_kernel, (B + 127) / 128, 128, 0, st, rs, B, t_row, t_pos, c_row, c_pos, G1);
    return cudaGetLastError();
}

template <typename T>
__global__ void __launch_bounds__(256) talker_embed_kernel(const RowState* __restrict__ rs, const T* __restrict__ cemb,
                                                           const T* __restrict__ pemb, int H, int V, int cpV, int G,
                                                           const int32_t* __restrict__ codes_ws, int frames_cap,
                                                           const float* __restrict__ text,
                                                           const float* __restrict__ pad, float* __restrict__ x,
                                                           int eos, int* err) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x;
    const RowState& s = rs[b];
    float* xr = x + (size_t)b * H;
    __shared__ int ids[MAX_GROUPS];
    __shared__ int ok;
    const float* trow = pad;
    if (s.finished) {
        if (threadIdx.x == 0) { ids[0] = eos; ok = 1; }
        __syncthreads();
        for (int i = threadIdx.x; i < H; i += 256) xr[i] = to_f(cemb[(size_t)eos * H + i]) + pad[i];
        return;
    }
    const int f = s.sel - 1;
    if (threadIdx.x < G) {
        ids[threadIdx.x] = codes_ws[((size_t)b * frames_cap + f) * MAX_GROUPS + threadIdx.x];
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int good = ids[0] >= 0 && ids[0] < V;
        for (int q = 1; q < G; ++q) good &= ids[q] >= 0 && ids[q] < cpV;
        ok = good;
        if (!good) atomicOr(err, ERRB_BOUNDS);
    }
    __syncthreads();
    if (!ok) {
        for (int i = threadIdx.x; i < H; i += 256) xr[i] = pad[i];
        return;
    }
    if (f < s.n_text) trow = text + (size_t)(s.text_off + f) * H;
    for (int i = threadIdx.x; i < H; i += 256) {
        float acc = to_f(cemb[(size_t)ids[0] * H + i]);
        for (int q = 1; q < G; ++q) acc += to_f(pemb[((size_t)(q - 1) * cpV + ids[q]) * H + i]);
        xr[i] = acc + trow[i];
    }
}

cudaError_t launch_talker_embed(int dtype, const RowState* rs, int B, const void* codec_emb, const void* cp_emb,
                                int H, int V, int cpV, int G, const int32_t* codes_ws, int frames_cap,
                                const float* text, const float* pad, float* x, int eos, int* err, cudaStream_t st) {
    if (dtype == Q3_BF16)
        launch_pdl(talker_embed_kernel<bf16>, B, 256, 0, st, rs, (const bf16*)codec_emb, (const bf16*)cp_emb, H, V, cpV, G,
                                                     codes_ws, frames_cap, text, pad, x, eos, err);
    else
        launch_pdl(talker_embed_kernel<float>, B, 256, 0, st, rs, (const float*)codec_emb, (const float*)cp_emb, H, V, cpV, G,
                                                      codes_ws, frames_cap, text, pad, x, eos, err);
    return cudaGetLastError();
}

template <typename T>
__global__ void __launch_bounds__(256) cp_embed_prefill_kernel(const RowState* __restrict__ rs,
                                                               const float* __restrict__ h,
                                                               const T* __restrict__ cemb, int H, int V,
                                                               int32_t* codes_ws, int frames_cap,
                                                               float* __restrict__ dst, int* err) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x;
    const RowState& s = rs[b];
    if (s.finished) return;
    const int f = s.sel - 1;
    const int c0 = s.code0;
    if (c0 < 0 || c0 >= V || f < 0 || f >= frames_cap) {
        if (threadIdx.x == 0) atomicOr(err, ERRB_BOUNDS);
        return;
    }
    if (threadIdx.x == 0) codes_ws[((size_t)b * frames_cap + f) * MAX_GROUPS] = c0;
    float* d0 = dst + (size_t)(2 * b) * H;
    float* d1 = d0 + H;
    for (int i = threadIdx.x; i < H; i += 256) {
        d0[i] = h[(size_t)b * H + i];
        d1[i] = to_f(cemb[(size_t)c0 * H + i]);
    }
}

cudaError_t launch_cp_embed_prefill(int dtype, RowState* rs, int B, const float* h, const void* codec_emb, int H,
                                    int V, int32_t* codes_ws, int frames_cap, float* dst, int* err, cudaStream_t st) {
    if (dtype == Q3_BF16)
        launch_pdl(cp_embed_prefill_kernel<bf16>, B, 256, 0, st, rs, h, (const bf16*)codec_emb, H, V, codes_ws, frames_cap,
                                                         dst, err);
    else
        launch_pdl(cp_embed_prefill_kernel<float>, B, 256, 0, st, rs, h, (const float*)codec_emb, H, V, codes_ws, frames_cap,
                                                          dst, err);
    return cudaGetLastError();
}

template <typename T>
__global__ void __launch_bounds__(256) cp_embed_step_kernel(const RowState* __restrict__ rs, const T* __restrict__ pemb,
                                                            int H, int cpV, int s_idx,
                                                            const int32_t* __restrict__ codes_ws, int frames_cap,
                                                            float* __restrict__ dst, int* err) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x;
    const RowState& s = rs[b];
    if (s.finished) return;
    const int f = s.sel - 1;
    const int c = codes_ws[((size_t)b * frames_cap + f) * MAX_GROUPS + s_idx];
    if (c < 0 || c >= cpV) {
        if (threadIdx.x == 0) atomicOr(err, ERRB_BOUNDS);
        return;
    }
    const T* src = pemb + ((size_t)(s_idx - 1) * cpV + c) * H;
    for (int i = threadIdx.x; i < H; i += 256) dst[(size_t)b * H + i] = to_f(src[i]);
}

cudaError_t launch_cp_embed_step(int dtype, const RowState* rs, int B, const void* cp_emb, int H, int cpV, int s,
                                 const int32_t* codes_ws, int frames_cap, float* dst, int* err, cudaStream_t st) {
    if (dtype == Q3_BF16)
        launch_pdl(cp_embed_step_kernel<bf16>, B, 256, 0, st, rs, (const bf16*)cp_emb, H, cpV, s, codes_ws, frames_cap, dst,
                                                      err);
    else
        launch_pdl(cp_embed_step_kernel<float>, B, 256, 0, st, rs, (const float*)cp_emb, H, cpV, s, codes_ws, frames_cap, dst,
                                                       err);
    return cudaGetLastError();
}

__global__ void pack_codes_kernel(const int32_t* __restrict__ ws, int frames_cap, long f0, int n, int G, int B,
                                  int32_t* __restrict__ dst, long pitch) {
    const long total = (long)B * n * G;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
        const int q = (int)(i % G);
        const long j = (i / G) % n;
        const int b = (int)(i / ((long)G * n));
        const long f = f0 + j;
        dst[(long)b * pitch + j * G + q] = f < frames_cap ? ws[((size_t)b * frames_cap + f) * MAX_GROUPS + q] : -1;
    }
}

cudaError_t launch_pack_codes(const int32_t* codes_ws, int frames_cap, long f0, int n, int G, int B, int32_t* dst,
                              long pitch, cudaStream_t st) {
    const long total = (long)B * n * G;
    if (total <= 0) return cudaSuccess;
    const int blocks = (int)std::min<long>((total + 255) / 256, 4096);
    pack_codes_kernel<<<blocks, 256, 0, st>>>(codes_ws, frames_cap, f0, n, G, B, dst, pitch);
    return cudaGetLastError();
}

}  // namespace q3

namespace q3 {

// ------------------------------------------------------------------ text side
// out[i][:] = emb[ids[i]][:] (fp32), one block per id; an id outside
// [0, vocab) leaves a zero row and sets the bounds bit.
template <typename T>
__global__ void __launch_bounds__(256) text_gather_kernel(const T* __restrict__ emb, const int32_t* __restrict__ ids,
                                                          int vocab, int width, float* __restrict__ out, int* err) {
    const int i = blockIdx.x;
    const int id = ids[i];
    const bool ok = id >= 0 && id < vocab;
    if (!ok && threadIdx.x == 0) atomicOr(err, ERRB_BOUNDS);
    for (int k = threadIdx.x; k < width; k += 256)
        out[(size_t)i * width + k] = ok ? to_f(emb[(size_t)id * width + k]) : 0.0f;
}

__global__ void silu_kernel(float* __restrict__ x, long n) {
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        const float v = x[i];
        x[i] = v / (1.0f + expf(-v));
    }
}

// SiLU(g) * u for the separate gate / up products, in place over g (the same
// expression as the stacked product's epilogue)
__global__ void silu_mul_kernel(float* __restrict__ g, const float* __restrict__ u, long n) {
    pdl_wait();
    pdl_trigger();
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        const float v = g[i];
        g[i] = v / (1.0f + expf(-v)) * u[i];
    }
}

cudaError_t launch_text_gather(int dtype, const void* emb, const int32_t* ids, int n, int vocab, int width, float* out,
                               int* err, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    if (dtype == Q3_BF16)
        text_gather_kernel<bf16><<<n, 256, 0, st>>>((const bf16*)emb, ids, vocab, width, out, err);
    else
        text_gather_kernel<float><<<n, 256, 0, st>>>((const float*)emb, ids, vocab, width, out, err);
    return cudaGetLastError();
}

cudaError_t launch_silu(float* x, long n, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    const int blocks = (int)std::min<long>((n + 255) / 256, 4L * device_sm_count());
    silu_kernel<<<blocks, 256, 0, st>>>(x, n);
    return cudaGetLastError();
}

cudaError_t launch_silu_mul(float* g, const float* u, long n, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    const int blocks = (int)std::min<long>((n + 255) / 256, 4L * device_sm_count());
    launch_pdl(silu_mul_kernel, blocks, 256, 0, st, g, u, n);
    return cudaGetLastError();
}

}  // namespace q3
