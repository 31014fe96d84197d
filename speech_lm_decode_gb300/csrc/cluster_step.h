// Parameters and host entry points of the cluster step kernel: one talker
// step of a single row (15 code-predictor passes with their draws, the
// talker input, 28 talker layers, codebook-0 selection) in one cooperative
// launch of eight thread-block clusters, one per KV head.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "q3tts.h"
#include "frame_params.h"

namespace q3 {

constexpr int CL_CS = 8;        // CTAs per cluster
constexpr int CL_NCL = 8;       // clusters (= KV heads)
constexpr int CL_NCTA = CL_CS * CL_NCL;
constexpr int CL_MAX_CP_LAYERS = 5;   // predictor layers whose K/V stay in shared memory

// Bytes of the packed weight image and the word buffers the kernel needs
// (0 when the configuration is not one the kernel serves).
struct ClLayout {
    size_t pack_bytes;     // packed weights (fragment order, per CTA slices)
    size_t xr_words;       // cross-cluster reduction words
    size_t lg_words;       // logit words (predictor and talker heads)
    // byte offsets inside the pack of each matrix class
    size_t off_t[4], off_c[4];   // per stack: QKV, O, GU, DOWN (layer 0; layers follow)
    size_t per_t[4], per_c[4];   // bytes per layer of each class (all CTAs)
    size_t off_cph, per_cph;     // predictor heads (head s at off + s * per)
    size_t off_th;               // talker codec head
    size_t off_proj;             // 1.7B-shaped projection into the predictor width
};

// Why the kernel cannot serve cfg ("" when it can).  Checks shapes only.
const char* cl_unsupported(const q3tts_config& c);
ClLayout cl_layout(const q3tts_config& c);

struct ClParams {
    const unsigned char* pack;
    ClLayout lay;
    // norms and the pieces read directly (fp32 norms; bf16 embeddings)
    const float* t_attn_norm; const float* t_q_norm; const float* t_k_norm; const float* t_mlp_norm;
    const float* t_final_norm;
    const float* c_attn_norm; const float* c_q_norm; const float* c_k_norm; const float* c_mlp_norm;
    const float* c_final_norm;
    const void* codec_emb;   // [V][H]
    const void* cp_emb;      // [G-1][cpV][H]
    const float* cp_proj_b;  // [Hc] or NULL
    int H, Hc, F, Fc, Lt, Lc, V, cpV, G, eos, sup_lo, sup_hi, max_batch, cap;
    float eps;
    const float2* rope;      // [rows][64] (cos, sin)
    void* Kc; void* Vc;      // talker cache [Lt][max_batch][8][cap][128] bf16 (row 0 used)
    RowState* rows;
    const q3tts_sampling* P;
    Word* xr;                // [2][NCL][2][2048] reduction words
    Word* lg;                // [2][cpV] predictor logits, then [V] talker logits
    float* h;                // talker post-norm hidden [H] (read by the next launch)
    int32_t* codes;          // [frames_cap][16]
    int frames_cap;
    const float* text;       // [n_text][H] of row 0
    const float* pad;
    unsigned* ctl;           // [0] abort flag
    int* err;
    float* cap_t; float* cap_c; const int* cap_slot; int cap_T;
    long long wait_ns;       // bound of every wait
    int inject_skip;         // test only: this reduction index is never written by CTA 0 (-1: off)
};

size_t cl_smem_bytes();
// One-time attribute setup and co-residency check: cudaSuccess when the
// 8 x 8 cooperative cluster launch fits this device.
cudaError_t cl_setup();
// Rearrange every bf16 matrix into the packed image (one launch per matrix).
cudaError_t cl_pack_weights(const q3tts_config& c, const q3tts_weights& w, unsigned char* pack, cudaStream_t st);
cudaError_t launch_cluster_step(const ClParams* params_dev, cudaStream_t st);

}  // namespace q3
