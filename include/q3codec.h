/*
 * q3codec.h -- C ABI of the GB300 (sm_103a) 12 Hz codec decoder: 16-code
 * frames -> 24 kHz waveform (1920 samples per frame).
 *
 * What it computes (ncnn port write-up "Qwen3-TTS 移植 ncnn 简明教程", ncnn
 * discussion 6798, section 1, Codec Decoder bullet): SplitRVQ dequantisation
 * (16 codebooks of 2048 x 256) -> an 8-layer transformer of width 512 with
 * head_dim 64, RoPE theta 1e4, a causal 72-frame window and LayerScale ->
 * 2 x (transposed convolution + ConvNeXt) -> a DAC-style vocoder (SnakeBeta
 * activations, upsampling 8, 5, 4, 3).  The decoder is causal end to end and
 * a request is decoded on a grid of 300-frame chunks, each with the 25 frames
 * before it as left context; streaming output decodes the current chunk
 * after the first 4 frames and then every 12 (Mizuoto "Qwen3-TTS" page,
 * section "速度").  Where the pages leave the structure open the library
 * takes these readings:
 *  - SplitRVQ: codebook 0 and codebooks 1..15 each sum their rows and have
 *    their own 256 -> 512 output projection (no bias); the two are added;
 *  - transformer layer: pre-norm RMSNorm, q/k/v/o without bias, rotate-half
 *    RoPE at the frame's index in the decoded window, attention over frames
 *    t-window+1..t, SiLU-gated MLP; each residual branch is multiplied by its
 *    LayerScale vector; a final RMSNorm;
 *  - upsampling stage: transposed convolution with kernel = stride = 2
 *    (bias), ConvNeXt block (causal depthwise conv width 7, LayerNorm,
 *    Linear -> exact GELU -> Linear, gamma, residual);
 *  - vocoder: causal Conv1d (k 7) to dac_channels, blocks of SnakeBeta +
 *    causal transposed convolution (kernel 2 x stride, trailing `stride`
 *    samples dropped) + 3 residual units (dilations 1, 3, 9: SnakeBeta, Conv
 *    k 7, SnakeBeta, Conv k 1), channels halving per block; SnakeBeta, Conv1d
 *    to one channel (k 7), tanh.  SnakeBeta(x) = x + sin^2(exp(a) x) /
 *    (exp(b) + 1e-9) per channel (log-scale a, b).
 *
 * Conventions as in q3tts.h (status codes, borrowed weights and workspace,
 * one synchronisation per call, host-or-device pointers, one stream per
 * handle, not thread-safe).  Weight layouts: Linear [out][in]; Conv1d
 * [Cout][K][Cin] (tap k multiplies x[t - (K-1-k) * dilation]); depthwise
 * [C][7] (fp32); transposed convolution [stride][Cout][K/stride][Cin], element
 * (r, co, j, ci) being kernel tap r + j * stride.  Matrices and convolution
 * kernels are in `dtype`; per-channel vectors (norms, biases, LayerScale,
 * gamma, SnakeBeta parameters) and the depthwise taps are fp32.
 */
#ifndef Q3CODEC_H
#define Q3CODEC_H

#include <stddef.h>
#include <stdint.h>

#include "q3tts.h"

#ifdef __cplusplus
extern "C" {
#endif

#define Q3C_MAX_BLOCKS 4

typedef struct {
    int n_codebooks;      /* 16 (codebook 0 = semantic)                          */
    int codebook_size;    /* 2048                                                */
    int codebook_dim;     /* 256                                                 */
    int hidden;           /* 512, transformer and upsampler width                */
    int n_layers;         /* 8                                                   */
    int n_heads;          /* 8; head_dim must be 64                              */
    int head_dim;
    int ffn;              /* SiLU-gated MLP width                                */
    int window;           /* 72: frames t-window+1..t are attended               */
    float rope_theta;     /* 1e4                                                 */
    float rms_eps;        /* RMSNorm epsilon                                     */
    float ln_eps;         /* ConvNeXt LayerNorm epsilon                          */
    int n_up;             /* x2 upsampling stages (2)                            */
    int up_ffn;           /* ConvNeXt MLP width                                  */
    int dac_channels;     /* vocoder width after its input convolution            */
    int n_blocks;         /* vocoder blocks (<= Q3C_MAX_BLOCKS)                  */
    int strides[Q3C_MAX_BLOCKS];
    int dtype;            /* Q3_F32 or Q3_BF16: matrices and convolution kernels */
    int max_frames;       /* longest window one call decodes (300 + 25 = 325)    */
    int tc_min_tokens;    /* rows from which products run on the tensor cores
                             (0: 16; negative: never)                            */
} q3codec_config;

/* Device pointers, borrowed; shapes with D = hidden, Dc = codebook_dim,
 * L = n_layers, U = n_up, F = ffn, F2 = up_ffn, C0 = dac_channels. */
typedef struct {
    const void* codebooks;    /* [16][2048][Dc]                                  */
    const void* proj_sem;     /* [D][Dc]                                         */
    const void* proj_ac;      /* [D][Dc]                                         */
    const void* attn_norm;    /* [L][D] fp32                                     */
    const void* wqkv;         /* [L][3D][D], rows q, k, v                        */
    const void* wo;           /* [L][D][D]                                       */
    const void* ls_attn;      /* [L][D] fp32                                     */
    const void* mlp_norm;     /* [L][D] fp32                                     */
    const void* wgu;          /* [L][2F][D], rows gate, up                       */
    const void* wd;           /* [L][D][F]                                       */
    const void* ls_mlp;       /* [L][D] fp32                                     */
    const void* final_norm;   /* [D] fp32                                        */
    const void* up_w;         /* [U][2][D][1][D]                                 */
    const void* up_b;         /* [U][D] fp32                                     */
    const void* dw_w;         /* [U][D][7] fp32                                  */
    const void* dw_b;         /* [U][D] fp32                                     */
    const void* ln_w;         /* [U][D] fp32                                     */
    const void* ln_b;         /* [U][D] fp32                                     */
    const void* fc1_w;        /* [U][F2][D]                                      */
    const void* fc1_b;        /* [U][F2] fp32                                    */
    const void* fc2_w;        /* [U][D][F2]                                      */
    const void* fc2_b;        /* [U][D] fp32                                     */
    const void* gamma;        /* [U][D] fp32                                     */
    const void* in_w;         /* [C0][7][D]                                      */
    const void* in_b;         /* [C0] fp32                                       */
    /* vocoder block b (Cin = C0 / 2^b, Cout = Cin / 2, s = strides[b]):
     * blk[b] = { snake a [Cin], snake b [Cin], transposed conv [s][Cout][2][Cin],
     *            its bias [Cout] }                                            */
    const void* blk[Q3C_MAX_BLOCKS][4];
    /* residual unit u of block b: { snake a1, b1 [Cout], conv [Cout][7][Cout],
     * bias [Cout], snake a2, b2 [Cout], conv [Cout][1][Cout], bias [Cout] }   */
    const void* unit[Q3C_MAX_BLOCKS][3][8];
    const void* out_a;        /* [C] fp32, C = last block's Cout                 */
    const void* out_b;        /* [C] fp32                                        */
    const void* out_w;        /* [1][7][C]                                       */
    const void* out_bias;     /* [1] fp32                                        */
} q3codec_weights;

typedef struct q3codec q3codec_t;

/* Workspace bytes for this configuration (0 if the configuration is invalid). */
size_t q3codec_workspace_bytes(const q3codec_config* cfg);

/* Bind a decoder to borrowed weights, a workspace of at least
 * q3codec_workspace_bytes() and a stream.  Errors: Q3_ERR_ARG (bad
 * configuration: head_dim != 64, widths not multiples of 8, channels that do
 * not halve evenly, NULL weight, small workspace), Q3_ERR_CUDA. */
int q3codec_create(const q3codec_config* cfg, const q3codec_weights* w, void* workspace, size_t ws_bytes,
                   void* stream, q3codec_t** out);

/* Samples per frame: 4 x the product of the strides (1920 at full size). */
int q3codec_samples_per_frame(const q3codec_t* h);

/* Decode one window of T frames (1 <= T <= max_frames) from a zero state and
 * write the samples of frames keep_from..T-1.  codes: [T][n_codebooks] int32,
 * host or device; wav: [(T - keep_from) * samples_per_frame] fp32, host or
 * device.  Errors: Q3_ERR_ARG (T, keep_from, NULL; a host code out of range),
 * Q3_ERR_BOUNDS (a device code out of range), Q3_ERR_CUDA. */
int q3codec_decode_window(q3codec_t* h, const int32_t* codes, int T, int keep_from, float* wav);

/* A whole request of T frames on the chunk grid: chunk c (frames 300c ..
 * 300c + 299) is decoded from frame max(0, 300c - 25) and its own frames'
 * samples are kept (requires max_frames >= min(T, 325)).  wav: [T *
 * samples_per_frame].  Errors as q3codec_decode_window. */
int q3codec_decode(q3codec_t* h, const int32_t* codes, int T, float* wav);

/* Streaming: q3codec_stream_reset() starts a request; q3codec_stream_push()
 * appends n frames (host codes [n][n_codebooks]) and, when a decode is due
 * (after the first 4 frames, then every 12 more, and at final != 0), decodes
 * the current chunk from its regular start and writes the samples not sent
 * before (finishing an earlier chunk first) to wav (host or device, room for
 * `capacity` samples); *n_samples receives how many.  The samples equal
 * q3codec_decode's up to rounding.  Errors: Q3_ERR_ARG, Q3_ERR_CAPACITY
 * (wav too small; nothing is consumed), Q3_ERR_STATE (push after final),
 * Q3_ERR_BOUNDS, Q3_ERR_CUDA. */
int q3codec_stream_reset(q3codec_t* h);
int q3codec_stream_push(q3codec_t* h, const int32_t* codes, int n, int final, float* wav, long capacity,
                        long* n_samples);

/* Kernels the last decoded window launched (for the benchmark's count). */
int q3codec_window_kernel_count(const q3codec_t* h);

const char* q3codec_last_error(const q3codec_t* h);
void q3codec_destroy(q3codec_t* h);

#ifdef __cplusplus
}
#endif
#endif
