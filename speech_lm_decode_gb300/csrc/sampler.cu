// Sampler kernels of the frame loop and the standalone test entry point; the
// processors and the draw themselves are in sampler.cuh.
#include "sampler.cuh"
#include "kernels.h"
#include "pdl.cuh"

namespace q3 {

size_t sampler_smem_bytes() { return sizeof(SampSmem); }

// ------------------------------------------------------------------ kernels
__global__ void __launch_bounds__(ST) talker_sample_kernel(const float* __restrict__ logits, int V, RowState* rs,
                                                           const q3tts_sampling* __restrict__ P, int eos, int sup_lo,
                                                           int sup_hi, int advance_pos, int* err, float* cap_logits,
                                                           const int* cap_slot, int cap_T) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) unsigned char smraw[];
    SampSmem& sm = *reinterpret_cast<SampSmem*>(smraw);
    const int b = blockIdx.x;
    RowState& s = rs[b];
    if (s.finished) return;
    const int k = s.sel;
    const q3tts_sampling p = P[b];
    const float* lg = logits + (size_t)b * V;
    if (cap_logits && cap_slot[b] >= 0 && k <= cap_T) {
        float* dst = cap_logits + ((size_t)cap_slot[b] * (cap_T + 1) + k) * V;
        for (int i = threadIdx.x; i < V; i += ST) dst[i] = lg[i];
    }
    const DrawCfg d{p.do_sample, p.temperature, p.top_k, p.top_p};
    int id = sample_row(sm, lg, V, d, true, p.repetition_penalty, s.seen, nullptr, k, p.min_new_tokens, eos, sup_lo,
                        sup_hi, p.seed, (uint32_t)b, (uint32_t)k, 0u);
    if (threadIdx.x == 0) {
        s.frames = k;
        if (id < 0) {
            atomicOr(err, ERRB_NAN);
            s.finished = 1;
            s.reason = Q3_FINISHED_ERROR;
            return;
        }
        if (p.force_eos_at_frame >= 0 && k == p.force_eos_at_frame) id = eos;
        if (id < MAX_VOCAB) s.seen[id >> 5] |= 1u << (id & 31);
        s.code0 = id;
        s.sel = k + 1;
        if (advance_pos) s.pos += 1;
        if (id == eos) { s.finished = 1; s.reason = Q3_FINISHED_EOS; }
        else if (k >= p.max_frames) { s.finished = 1; s.reason = Q3_FINISHED_LENGTH; }
    }
}

__global__ void __launch_bounds__(ST) cp_sample_kernel(const float* __restrict__ logits, int V, RowState* rs,
                                                       const q3tts_sampling* __restrict__ P, int s_idx,
                                                       int32_t* codes_ws, int frames_cap, int* err, float* cap_logits,
                                                       const int* cap_slot, int cap_T, int G) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) unsigned char smraw[];
    SampSmem& sm = *reinterpret_cast<SampSmem*>(smraw);
    const int b = blockIdx.x;
    RowState& s = rs[b];
    if (s.finished) return;
    const int f = s.sel - 1;
    const q3tts_sampling p = P[b];
    const float* lg = logits + (size_t)b * V;
    if (cap_logits && cap_slot[b] >= 0 && f < cap_T) {
        float* dst = cap_logits + (((size_t)cap_slot[b] * cap_T + f) * (G - 1) + s_idx) * V;
        for (int i = threadIdx.x; i < V; i += ST) dst[i] = lg[i];
    }
    const DrawCfg d{p.cp_do_sample, p.cp_temperature, p.cp_top_k, p.cp_top_p};
    const int id = sample_row(sm, lg, V, d, false, 1.0f, nullptr, nullptr, 0, 0, -1, 0, 0, p.seed, (uint32_t)b,
                              (uint32_t)f, (uint32_t)(s_idx + 1));
    if (threadIdx.x == 0) {
        if (id < 0) {
            atomicOr(err, ERRB_NAN);
            s.finished = 1;
            s.reason = Q3_FINISHED_ERROR;
            s.frames = f;
            return;
        }
        codes_ws[((size_t)b * frames_cap + f) * MAX_GROUPS + s_idx + 1] = id;
    }
}

__global__ void __launch_bounds__(ST) sample_sets_kernel(const float* __restrict__ logits, int V, int talker,
                                                         const q3tts_sampling* __restrict__ P,
                                                         const uint8_t* __restrict__ seen,
                                                         const int32_t* __restrict__ sel_index, int step,
                                                         const int32_t* __restrict__ noise_row, int eos, int sup_lo,
                                                         int sup_hi, int32_t* ids, int* err) {
    extern __shared__ __align__(16) unsigned char smraw[];
    SampSmem& sm = *reinterpret_cast<SampSmem*>(smraw);
    const int b = blockIdx.x;
    const q3tts_sampling p = P[b];
    const DrawCfg d = talker ? DrawCfg{p.do_sample, p.temperature, p.top_k, p.top_p}
                             : DrawCfg{p.cp_do_sample, p.cp_temperature, p.cp_top_k, p.cp_top_p};
    const int id = sample_row(sm, logits + (size_t)b * V, V, d, talker != 0, p.repetition_penalty, nullptr,
                              seen ? seen + (size_t)b * V : nullptr, sel_index[b], talker ? p.min_new_tokens : 0,
                              talker ? eos : -1, talker ? sup_lo : 0, talker ? sup_hi : 0, p.seed,
                              (uint32_t)noise_row[b], (uint32_t)sel_index[b], (uint32_t)step);
    if (threadIdx.x == 0) {
        ids[b] = id;
        if (id < 0) atomicOr(err, ERRB_NAN);
    }
}

cudaError_t sampler_init() {
    const int bytes = (int)sizeof(SampSmem);
    cudaError_t e = cudaFuncSetAttribute(talker_sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(cp_sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(sample_sets_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return e;
}

cudaError_t launch_talker_sample(const float* logits, int V, int B, RowState* rs, const q3tts_sampling* P, int eos,
                                 int sup_lo, int sup_hi, int advance_pos, int* err, float* cap_logits,
                                 const int* cap_slot, int cap_T, cudaStream_t st) {
    launch_pdl(talker_sample_kernel, B, ST, sizeof(SampSmem), st, logits, V, rs, P, eos, sup_lo, sup_hi, advance_pos, err,
                                                          cap_logits, cap_slot, cap_T);
    return cudaGetLastError();
}

cudaError_t launch_cp_sample(const float* logits, int V, int B, RowState* rs, const q3tts_sampling* P, int s,
                             int32_t* codes_ws, int frames_cap, int* err, float* cap_logits, const int* cap_slot,
                             int cap_T, int n_groups, cudaStream_t st) {
    launch_pdl(cp_sample_kernel, B, ST, sizeof(SampSmem), st, logits, V, rs, P, s, codes_ws, frames_cap, err, cap_logits,
                                                      cap_slot, cap_T, n_groups);
    return cudaGetLastError();
}

cudaError_t launch_sample_sets(const float* logits, int n, int V, int talker, const q3tts_sampling* P,
                               const uint8_t* seen, const int32_t* sel_index, int step, const int32_t* noise_row,
                               int eos, int sup_lo, int sup_hi, int32_t* ids, int* err, cudaStream_t st) {
    sample_sets_kernel<<<n, ST, sizeof(SampSmem), st>>>(logits, V, talker, P, seen, sel_index, step, noise_row, eos,
                                                        sup_lo, sup_hi, ids, err);
    return cudaGetLastError();
}

}  // namespace q3
