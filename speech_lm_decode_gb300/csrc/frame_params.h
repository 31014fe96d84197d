// Parameters of the persistent frame kernel (filled on the host, read on the device).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "q3tts.h"

namespace q3 {

struct RowState;

struct PBlk {
    const float* attn_norm;
    const void* wqkv;
    const float* q_norm;
    const float* k_norm;
    const void* wo;
    const float* mlp_norm;
    const void* wgu;
    const void* wd;
    const float* final_norm;
    void* Kc;
    void* Vc;
    int cap, L, H, F;
};

struct FrameParams {
    PBlk t, c;
    const void* codec_emb;
    const void* codec_head;
    const void* cp_emb;
    const void* cp_heads;
    const void* cp_proj_w;
    const float* cp_proj_b;
    int H, Hc, V, cpV, G, nq, nkv, eos, sup_lo, sup_hi, n_splits, kmax, max_batch;
    float eps;
    const float2* rope;
    int rope_rows;
    RowState* rows;
    const q3tts_sampling* P;
    float* x;       // talker residual [H]
    float* cx;      // predictor residual [2][Hc]
    float* h;       // talker post-norm hidden [H]
    float* qkv;     // [2][nqkv]
    float* part;    // attention partials [2][nkv][S][GQ][HD+2]
    float* o;       // attention output operand [2][nq*HD]
    float* act;     // SiLU(g)*u operand [2][F]
    float* logits;  // [V]
    float* cpl;     // [cpV]
    int32_t* codes;
    int frames_cap;
    const float* text;
    const float* pad;
    unsigned* bar;    // [0] grid barrier counter; [1] abort flag; [2..] per-head split counters
                      // (zeroed before every launch)
    int* err;
    float* cap_t;
    float* cap_c;
    const int* cap_slot;
    int cap_T;
    int xin_bytes;    // shared-memory bytes of the input-vector region
};


constexpr int FRAME_BAR_WORDS = 64;

// Shared memory the frame kernel needs with an input-vector region of
// xin_bytes (0 if it does not fit one SM); the attention scratch that shares
// that region needs frame_attn_scratch_bytes().
size_t frame_smem_bytes(int dtype, int xin_bytes);
size_t frame_attn_scratch_bytes();
// One-time attribute setup; returns cudaSuccess when the kernel can run.
cudaError_t frame_setup(int dtype, size_t smem);
// CTAs of the frame kernel that fit one SM with this shared memory.
cudaError_t frame_occupancy(int dtype, size_t smem, int* blocks);
// Launch one talker step (cooperative, one CTA per SM).
cudaError_t launch_frame(int dtype, const FrameParams* params_dev, int grid, size_t smem, cudaStream_t st);

}  // namespace q3
