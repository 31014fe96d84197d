// Host-callable launchers of the q3tts kernels.  Every launcher enqueues on
// `st` and returns the launch status (cudaGetLastError).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "q3tts.h"

namespace q3 {

struct RowState;

// SMs of the current device (looked up once per device).
int device_sm_count();

// Launch `k` allowing programmatic dependent launch (it may overlap the tail of
// the previous kernel in the stream); `k` must start with pdl_wait().
template <typename... K, typename... A>
inline cudaError_t launch_pdl(void (*k)(K...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, A&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, static_cast<A&&>(args)...);
}

// The draw settings every selection needs: temperature > 0 where the draw
// samples, and (talker chain) a positive repetition penalty.
inline bool sampling_ok(const q3tts_sampling& s, bool talker) {
    if (talker) return (!s.do_sample || s.temperature > 0.f) && s.repetition_penalty > 0.f;
    return !s.cp_do_sample || s.cp_temperature > 0.f;
}

// ---------------------------------------------------------------- linear.cu
// Scratch of the tensor-core path: the fp32 operand split into bf16 high and
// low parts ([M][K] each).
struct TcScratch {
    void* base = nullptr;
    size_t bytes = 0;
    int min_tokens = 16;   // tokens from which the tensor-core path runs (<= 0: never)
};
inline bool tc_fits(const TcScratch& s, int M, int K) { return s.base && (size_t)M * K * 4 <= s.bytes; }
// true when launch_linear / launch_linear_gated over M tokens of width K take
// the tensor-core path, whose operand can then be written pre-split (X = NULL)
bool linear_takes_split(int dtype, int M, int K, const TcScratch& tc);

// Y[m][n] (+)= sum_k W[n][k] X[m][k] (+ bias[n]); W [N][K] in the model dtype,
// X [M][K] fp32 (leading dimension ldx), Y fp32 (leading dimension ldy).
// accumulate: add into Y (residual).  X = NULL: the operand is already in the
// tensor-core scratch as bf16 high / low parts (only where linear_takes_split;
// cudaErrorInvalidValue otherwise).
cudaError_t launch_linear(int dtype, const void* W, int N, int K, const float* X, int ldx, int M, float* Y, int ldy,
                          const float* bias, int accumulate, const TcScratch& tc, int* err, cudaStream_t st);
// SwiGLU projection: out[m][n] = silu(g) * u with g = W[n].x, u = W[F+n].x,
// W [2F][K]; out fp32 with leading dimension ldo, or (out_split != NULL, only
// where linear_takes_split) the bf16 high / low parts [M][F] in out_split,
// the operand of a following launch_linear(X = NULL) on that scratch.
cudaError_t launch_linear_gated(int dtype, const void* W, int F, int K, const float* X, int ldx, int M, float* out,
                                int ldo, const TcScratch& tc, int* err, cudaStream_t st,
                                const TcScratch* out_split = nullptr);
// tensor-core (tcgen05) variants for bf16 weights and many tokens (gemm_tc.cu)
bool tc_available();
cudaError_t launch_linear_tc(const void* W, int N, int K, const float* X, int ldx, int M, float* Y, int ldy,
                             const float* bias, int accumulate, const TcScratch& tc, int* err, cudaStream_t st);
cudaError_t launch_linear_gated_tc(const void* W, int F, int K, const float* X, int ldx, int M, float* out, int ldo,
                                   const TcScratch& tc, int* err, cudaStream_t st,
                                   const TcScratch* out_split = nullptr);
// out[row(m)] = x[m] * rsqrt(mean(x[m]^2) + eps) * w; optionally hout (a
// second copy).  out_row: NULL = identity, else the output row of each input
// row (negative: skip).
cudaError_t launch_rmsnorm(const float* x, int ldx, int M, const float* w, int n, float eps, float* out, int ldo,
                           float* hout, int ldh, const int* out_row, cudaStream_t st);
// The same normalized rows written straight into the tensor-core scratch as
// bf16 high and low parts ([M][n] each: high = bf16(y), low = bf16(y - high)),
// the operand launch_linear(X = NULL) expects.
cudaError_t launch_rmsnorm_split(const float* x, int ldx, int M, const float* w, int n, float eps,
                                 const TcScratch& tc, cudaStream_t st);

// ---------------------------------------------------------------- attention.cu
// Per token m (row tok_row[m], position tok_pos[m] >= 0): per-head RMSNorm of
// q and k, RoPE at the position, q written back in place, k and v appended to
// the layer's cache [maxB][nkv][cap][128].  tok_pos < 0: token skipped.
cudaError_t launch_qk_rope_kv(int dtype, float* qkv, int ldq, int M, int nq, int nkv, const float* q_norm,
                              const float* k_norm, float eps, const float* rope_cs, int rope_rows, void* Kc, void* Vc,
                              int cap, const int* tok_row, const int* tok_pos, int* err, cudaStream_t st);
// Split-KV grouped-query decode attention over positions 0..tok_pos[m] of the
// token's row, then (n_splits > 1) the combine, writing the O-projection
// operand [M][nq*128]: fp32 into out, or (split != NULL) as the bf16 high /
// low parts the tensor-core projection reads with X = NULL.  bf16 caches with
// two q heads per kv head stream the cache through shared memory with bulk
// copies; a wait that runs out there sets the TIMEOUT bit of err.
cudaError_t launch_attention(int dtype, const float* qkv, int ldq, int M, int nq, int nkv, const void* Kc,
                             const void* Vc, int cap, const int* tok_row, const int* tok_pos, int n_splits,
                             float* part_m, float* part_l, float* part_acc, float* out, int ldo, int* err,
                             cudaStream_t st, const TcScratch* split = nullptr);

// Decode step over short bf16 caches (cap <= 64, two q heads per kv head)
// with QK-norm, RoPE and the K/V append of launch_qk_rope_kv fused in; every
// token of the launch must belong to a different row.  Output as in
// launch_attention.
cudaError_t launch_attention_short_fused(const float* qkv, int ldq, int M, int nq, int nkv, const float* q_norm,
                                         const float* k_norm, float eps, const float* rope_cs, int rope_rows,
                                         void* Kc, void* Vc, int cap, const int* tok_row, const int* tok_pos,
                                         float* out, int ldo, int* err, cudaStream_t st,
                                         const TcScratch* split = nullptr);

// Causal attention of prompt tokens, tiled: tiles[t] = {first token, tokens
// (1..64, consecutive positions of one row), row, position of the first};
// every token of a tile attends to positions 0..its own of its row's cache
// (bf16 caches: K / V enter the tensor cores exactly).  Output as in
// launch_attention (fp32 into out, or the bf16 high / low split).
cudaError_t launch_prefill_attention(int dtype, const float* qkv, int ldq, int M, int nq, int nkv, const void* Kc,
                                     const void* Vc, int cap, const int4* tiles, int n_tiles, float* out, int ldo,
                                     cudaStream_t st, const TcScratch* split = nullptr);

// ---------------------------------------------------------------- sampler.cu
size_t sampler_smem_bytes();
cudaError_t sampler_init();
// Talker selection for every unfinished row of the batch (see q3tts.h).
cudaError_t launch_talker_sample(const float* logits, int V, int B, RowState* rs, const q3tts_sampling* P, int eos,
                                 int sup_lo, int sup_hi, int advance_pos, int* err, float* cap_logits,
                                 const int* cap_slot, int cap_T, cudaStream_t st);
// Predictor draw s (0..14) -> codebook s+1 of frame sel-1, for unfinished rows.
cudaError_t launch_cp_sample(const float* logits, int V, int B, RowState* rs, const q3tts_sampling* P, int s,
                             int32_t* codes_ws, int frames_cap, int* err, float* cap_logits, const int* cap_slot,
                             int cap_T, int n_groups, cudaStream_t st);
// Standalone processors + draw on given logit sets.
cudaError_t launch_sample_sets(const float* logits, int n, int V, int talker, const q3tts_sampling* P,
                               const uint8_t* seen, const int32_t* sel_index, int step, const int32_t* noise_row,
                               int eos, int sup_lo, int sup_hi, int32_t* ids, int* err, cudaStream_t st);

// ---------------------------------------------------------------- loop.cu
cudaError_t launch_prepare_step(RowState* rs, int B, int* t_row, int* t_pos, int* c_row, int* c_pos, int G1,
                                cudaStream_t st);
cudaError_t launch_talker_embed(int dtype, const RowState* rs, int B, const void* codec_emb, const void* cp_emb,
                                int H, int V, int cpV, int G, const int32_t* codes_ws, int frames_cap,
                                const float* text, const float* pad, float* x, int eos, int* err, cudaStream_t st);
// Predictor prefill tokens [h, codec_emb(code0)] -> dst rows 2b, 2b+1 (width
// H); also writes codes_ws[b][f][0] = code0.
cudaError_t launch_cp_embed_prefill(int dtype, RowState* rs, int B, const float* h, const void* codec_emb, int H,
                                    int V, int32_t* codes_ws, int frames_cap, float* dst, int* err, cudaStream_t st);
// Predictor step s (1..14) token table[s-1](code_s) -> dst row b (width H).
cudaError_t launch_cp_embed_step(int dtype, const RowState* rs, int B, const void* cp_emb, int H, int cpV, int s,
                                 const int32_t* codes_ws, int frames_cap, float* dst, int* err, cudaStream_t st);

// Text side: out[i] = emb[ids[i]] as fp32 rows of `width` (a zero row and the
// bounds bit for an id outside [0, vocab)); x = SiLU(x) over n values.
cudaError_t launch_text_gather(int dtype, const void* emb, const int32_t* ids, int n, int vocab, int width, float* out,
                               int* err, cudaStream_t st);
cudaError_t launch_silu(float* x, long n, cudaStream_t st);
// g[m][f] = silu(g[m][f]) * u[m][f] for the separate gate / up products
// (g and u [M][F] fp32 with leading dimension F).
cudaError_t launch_silu_mul(float* g, const float* u, long n, cudaStream_t st);

// dst[b*pitch + j*G + q] = codes of frame f0+j of row b (-1 past the buffer).
cudaError_t launch_pack_codes(const int32_t* codes_ws, int frames_cap, long f0, int n, int G, int B, int32_t* dst,
                              long pitch, cudaStream_t st);

}  // namespace q3
