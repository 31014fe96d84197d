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

// Activations exchanged between CTAs of one launch are 64-bit words: the fp32
// value in the low half and the epoch of the phase that wrote it in the high
// half, so a reader knows from the word itself that it is current.
using Word = unsigned long long;

struct FrameParams {
    PBlk t, c;
    const void* codec_emb;
    const void* codec_head;
    const void* cp_emb;
    const void* cp_heads;
    const void* cp_proj_w;
    const float* cp_proj_b;
    int H, Hc, V, cpV, G, nq, nkv, eos, sup_lo, sup_hi, n_splits, max_batch;
    float eps;
    const float2* rope;
    int rope_rows;
    RowState* rows;
    const q3tts_sampling* P;
    Word* x;        // talker residual [H]
    Word* cx;       // predictor residual [2][Hc]
    Word* qkv;      // [2][(nq + 2 nkv) * 128]
    Word* o;        // attention output [2][nq * 128]
    Word* act;      // SiLU(g) * u [2][F]
    Word* logits;   // talker logits [V]
    Word* cpl;      // predictor logits [cpV]
    float* h;       // talker post-norm hidden [H] (read by the next launch)
    float* part;    // attention partials
    int32_t* codes;
    int frames_cap;
    const float* text;
    const float* pad;
    unsigned* ctl;  // [0] abort flag (sticky until the next prefill clears it);
                    // [8 + g] split counter of kv head g (talker attention)
    int* err;
    float* cap_t;
    float* cap_c;
    const int* cap_slot;
    int cap_T;
    int xin_bytes;  // shared-memory bytes of the attention scratch region
    long long wait_cycles;  // SM cycles before a device wait gives up
    unsigned inject_ep;     // test only: waits for words of this epoch never end (0: none)
};

constexpr int FRAME_CTL_WORDS = 64;
constexpr int FRAME_MAX_ROWS = 128;   // residual rows one CTA updates in one phase
constexpr int FRAME_MAX_PART = 1024;  // partial sums of one phase on one CTA (rows x 2 x 2 x 8 splits)
constexpr int FRAME_MAX_PHASES = 1024;  // phases of one launch (epoch = selection * 1024 + phase)
constexpr int FRAME_MAX_NORM = 2048;    // widest RMSNorm input (talker and predictor widths)

// Shared memory the frame kernel needs with an attention scratch region of
// xin_bytes (at least frame_attn_scratch_bytes()); 0 if it does not fit one SM.
// tc_rows: bf16 GEMV rows on the tensor cores (else FMA rows)
size_t frame_smem_bytes(int dtype, int xin_bytes, bool tc_rows);
size_t frame_attn_scratch_bytes();
// bytes of one weight ring slot of a kernel variant
size_t frame_tile_bytes(bool tc_rows);
constexpr int FRAME_CP_VMAX = 2048;   // largest predictor vocabulary the frame kernel draws over
// One-time attribute setup; returns cudaSuccess when the kernel can run.
cudaError_t frame_setup(int dtype, size_t smem, bool tc_rows);
// CTAs of the frame kernel that fit one SM with this shared memory.
cudaError_t frame_occupancy(int dtype, size_t smem, bool tc_rows, int* blocks);
// Launch one talker step (cooperative, `grid` CTAs).
cudaError_t launch_frame(int dtype, bool tc_rows, const FrameParams* params_dev, int grid, size_t smem,
                         cudaStream_t st);

}  // namespace q3
