/*
 * q3tts.h -- C ABI of the GB300 (sm_103a) Qwen3-TTS 12 Hz frame loop.
 *
 * One 80 ms frame of speech is 16 codec codes.  It is produced by one step of
 * the talker (a 28-layer Qwen3 decoder with a 3072-way codec head, which picks
 * codebook 0) followed by the code predictor (5 layers, 15 embedding tables
 * and 15 heads, which fill codebooks 1..15).  The next talker input is the sum
 * of the 16 code embeddings plus the trailing text embedding.  Sources: the
 * ncnn port write-up "Qwen3-TTS 移植 ncnn 简明教程" (ncnn discussion 6798),
 * section 1 "先搞清楚结构"; the strict-parity port (ncnn discussion 6832),
 * sections 3.1-3.2; the Mizuoto "Qwen3-TTS" engine page, sections
 * "工作原理", "与上游一致的做法" and "速度".
 *
 * Conventions shared by every entry point
 *  - Return value: Q3_OK (0) or one of the Q3_ERR_* codes; q3tts_last_error()
 *    gives a one-line reason.  Arguments are validated on the host before any
 *    work is queued.  Device-side failures (NaN logits, out-of-range ids) are
 *    recorded in a device error word and reported by the call that reads it:
 *    every call ends with exactly one synchronisation of the handle's stream.
 *  - Ownership: weights and the workspace are BORROWED device memory.  The
 *    caller allocates them, keeps them alive and unmodified until
 *    q3tts_destroy(), and frees them afterwards.  The library never allocates
 *    device memory itself; the static KV caches, per-row state and
 *    activations all live in the workspace.  Host arrays passed to a call are
 *    read (or written) during that call only.
 *  - Pointers documented as "host or device" may be either; the library asks
 *    the CUDA runtime which one it was given and copies as needed.
 *  - Layouts are row-major, C order.  Matrices are [out_features][in_features].
 *  - A handle is bound to one CUDA stream and is not thread-safe.
 */
#ifndef Q3TTS_H
#define Q3TTS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define Q3_OK            0
#define Q3_ERR_ARG       1  /* invalid argument, shape or id; nothing was queued        */
#define Q3_ERR_CUDA      2  /* a CUDA runtime call failed                                */
#define Q3_ERR_CAPACITY  3  /* prompt + frames would exceed max_ctx, or batch > max      */
#define Q3_ERR_STATE     4  /* call out of order (e.g. step before prefill)             */
#define Q3_ERR_NAN       5  /* NaN or +inf logits at a selection (fails closed)         */
#define Q3_ERR_TIMEOUT   6  /* a bounded device-side wait gave up                       */
#define Q3_ERR_BOUNDS    7  /* a device-side id or position check failed                */

/* weight / KV-cache element types */
#define Q3_F32   0
#define Q3_BF16  1

/* per-row finish reasons */
#define Q3_RUNNING          0
#define Q3_FINISHED_EOS     1  /* codebook 0 selected EOS (or a forced EOS)             */
#define Q3_FINISHED_LENGTH  2  /* max_frames frames completed without EOS               */
#define Q3_FINISHED_ERROR   3  /* the row's logits held NaN / +inf                      */

/* Model shape and sizing.  Every dimension and special id is explicit; there
 * are no hidden defaults (the checkpoint's config.json is authoritative on the
 * pages: eos 2150, not a code default).  Constraints: head_dim == 128,
 * n_q_heads a multiple of n_kv_heads, hidden/ffn/cp_hidden/cp_ffn multiples of
 * 8, n_groups <= 16, codec_vocab <= 4096, cp_vocab <= 4096. */
typedef struct {
    int n_layers;       /* talker layers (28)                                  */
    int hidden;         /* talker width H (1024 for 0.6B, 2048 for 1.7B)       */
    int n_q_heads;      /* 16                                                  */
    int n_kv_heads;     /* 8                                                   */
    int head_dim;       /* 128                                                 */
    int ffn;            /* talker SwiGLU width F                               */
    int codec_vocab;    /* 3072: codes 0..2047, specials above                 */
    int cp_layers;      /* predictor layers (5)                                */
    int cp_hidden;      /* predictor width (1024)                              */
    int cp_ffn;         /* predictor SwiGLU width                              */
    int cp_vocab;       /* 2048                                                */
    int n_groups;       /* codebooks per frame (16)                            */
    int eos_id;         /* 2150                                                */
    int suppress_lo;    /* 2048: ids [suppress_lo, suppress_hi) except eos     */
    int suppress_hi;    /* 3072      are masked at talker selections           */
    float rms_eps;      /* 1e-6                                                */
    float rope_theta;   /* 1e6                                                 */
    int dtype;          /* Q3_F32 or Q3_BF16: weights and KV cache             */
    int max_batch;      /* rows per handle                                     */
    int max_ctx;        /* talker positions per row (prompt + frames)          */
    int max_text;       /* trailing text rows per row                          */
    /* Execution choices (all explicit; 0 selects the documented default).    */
    int step_path;      /* batch-1 step: Q3_PATH_AUTO (the single-launch frame
                           kernel where the shape allows, else per-layer
                           kernels), or one path forced: Q3_PATH_GRAPH,
                           Q3_PATH_FRAME, Q3_PATH_CLUSTER (create fails with
                           Q3_ERR_ARG if it cannot serve)                      */
    int tc_min_tokens;  /* tokens from which projections run as tcgen05 GEMMs
                           (0: 16; negative: never)                            */
    int debug_sync;     /* 1: wait for every launch outside graph capture and
                           report it on stderr (diagnostics, slow)             */
    int wait_limit_us;  /* bound of every device-side wait of the batch-1
                           kernels, microseconds (0: 2,000,000)                */
    int inject_timeout; /* test only (0 = off).  Frame kernel: the readers of
                           phase n of the first step after a prefill wait for
                           an epoch no phase writes (n < 1024).  Cluster
                           kernel: the cross-cluster exchange with index n is
                           never written by CTA 0.  Every wait on it runs out
                           and the step returns Q3_ERR_TIMEOUT                 */
    int text_vocab;     /* text side (q3tts_text_embed): BPE vocabulary
                           (151936 upstream); 0 = no text path                */
    int text_hidden;    /* width of the text embedding (2048)                 */
    int separate_projections; /* 1: q, k, v and gate, up as separate products
                           (the layout of a model loaded without stacking,
                           Mizuoto "Qwen3-TTS" page, section "速度", fast mode
                           off); 0: stacked q/k/v and gate/up weights in one
                           product each.  The weights are the same stacked
                           arrays either way.  Per-layer kernels only (batch
                           > 1, prefill, Q3_PATH_GRAPH); every output row is
                           the same dot product in both, so results differ
                           only where the tensor-core tile / K-split choice,
                           which depends on the product's width, differs      */
} q3tts_config;

/* step_path values */
#define Q3_PATH_AUTO     0
#define Q3_PATH_GRAPH    1  /* per-layer kernels replayed as a CUDA graph        */
#define Q3_PATH_FRAME    2  /* one cooperative launch, epoch-tagged exchange words */
#define Q3_PATH_CLUSTER  3  /* one cooperative launch of 8 x 8 thread-block
                               clusters (one per KV head)                         */

/* One decoder stack (talker or predictor), layer-stacked, device pointers.
 * Norm weights are fp32; matrices are in the config dtype. */
typedef struct {
    const void* attn_norm;   /* [L][H]        f32                                   */
    const void* wqkv;        /* [L][(nq+2nkv)*hd][H]  rows: q heads, k heads, v heads */
    const void* q_norm;      /* [L][hd]       f32 (shared by all q heads)           */
    const void* k_norm;      /* [L][hd]       f32                                   */
    const void* wo;          /* [L][H][nq*hd]                                       */
    const void* mlp_norm;    /* [L][H]        f32                                   */
    const void* wgu;         /* [L][2F][H]    rows: gate 0..F-1, then up 0..F-1     */
    const void* wd;          /* [L][H][F]                                           */
    const void* final_norm;  /* [H]           f32                                   */
} q3tts_block_weights;

typedef struct {
    q3tts_block_weights talker;
    const void* codec_emb;   /* [codec_vocab][H]            talker codec embedding   */
    const void* codec_head;  /* [codec_vocab][H]                                     */
    q3tts_block_weights cp;  /* predictor stack, width cp_hidden                     */
    const void* cp_emb;      /* [n_groups-1][cp_vocab][H]   table q-1 embeds code q  */
    const void* cp_heads;    /* [n_groups-1][cp_vocab][cp_hidden] head s -> code s+1 */
    const void* cp_proj_w;   /* [cp_hidden][H] or NULL when H == cp_hidden           */
    const void* cp_proj_b;   /* [cp_hidden] f32 or NULL                              */
    /* text side, NULL when config.text_vocab == 0: embedding and ResizeMLP
     * (text_hidden -> text_hidden -> H with SiLU between the two layers)     */
    const void* text_emb;    /* [text_vocab][text_hidden]                            */
    const void* text_fc1_w;  /* [text_hidden][text_hidden]                           */
    const void* text_fc1_b;  /* [text_hidden] f32                                    */
    const void* text_fc2_w;  /* [H][text_hidden]                                     */
    const void* text_fc2_b;  /* [H] f32                                              */
} q3tts_weights;

/* Per-row generation settings (talker and predictor draws). */
typedef struct {
    int do_sample;            /* 0: greedy argmax (lowest index wins ties)           */
    float temperature;        /* > 0                                                 */
    int top_k;                /* <= 0: off                                           */
    float top_p;              /* >= 1: off                                           */
    float repetition_penalty; /* over this row's earlier codebook-0 selections       */
    int min_new_tokens;       /* EOS logit is -inf at selections 0..min_new-1        */
    uint64_t seed;            /* key of the counter-based noise                      */
    int max_frames;           /* the row ends on length after this many frames       */
    int force_eos_at_frame;   /* selection k == this becomes EOS; -1: never          */
    int cp_do_sample;         /* predictor draws: no penalty / suppression / min_new */
    float cp_temperature;
    int cp_top_k;
    float cp_top_p;
} q3tts_sampling;

typedef struct q3tts q3tts_t;

/* Bytes of device workspace a handle needs for this configuration
 * (0 if the configuration is invalid). */
size_t q3tts_workspace_bytes(const q3tts_config* cfg);

/* Create a handle.  cfg, w: read during the call.  workspace: device memory of
 * at least q3tts_workspace_bytes(cfg) bytes, 256-byte aligned, borrowed.
 * stream: a cudaStream_t (NULL = legacy default stream).  Errors: Q3_ERR_ARG
 * (bad shape, NULL weight, small workspace), Q3_ERR_CUDA. */
int q3tts_create(const q3tts_config* cfg, const q3tts_weights* w, void* workspace, size_t workspace_bytes,
                 void* stream, q3tts_t** out);

/* Prompt prefill and selection 0 of every row (Mizuoto page "与上游一致的做法":
 * the codec head reads the prefill's last position; ncnn discussion 6832 3.1:
 * step 0 only selects the first codebook-0 id).
 *   batch           rows, 1..max_batch
 *   prompt          [sum(len)][H] f32, host or device: row r is
 *                   rows prompt_offsets[r] .. prompt_offsets[r+1]-1
 *   prompt_offsets  [batch+1] host, non-decreasing, len >= 1 per row
 *   text            [sum(n_text)][H] f32, host or device (NULL if all empty):
 *                   trailing text rows, one consumed per talker step
 *   text_offsets    [batch+1] host
 *   tts_pad         [H] f32, host or device: used once a row's text runs out
 *   rows            [batch] host: per-row settings
 *   code0_out       [batch] int32, host or device, or NULL: selection 0
 * Resets every row.  Errors: Q3_ERR_ARG, Q3_ERR_CAPACITY (len + max_frames >
 * max_ctx, n_text > max_text), Q3_ERR_NAN, Q3_ERR_CUDA. */
int q3tts_prefill(q3tts_t* h, int batch, const float* prompt, const int32_t* prompt_offsets, const float* text,
                  const int32_t* text_offsets, const float* tts_pad, const q3tts_sampling* rows,
                  int32_t* code0_out);

/* Run n_frames talker steps on every unfinished row (ncnn discussion 6832 3.1:
 * step k > 0 consumes the pending codebook-0 id, completes frame k-1 through
 * the code predictor and selects the next id; N frames take N+1 selections).
 *   codes_out       [batch][n_frames][n_groups] int32, host or device, or NULL:
 *                   frames completed by this call, in call order (frame index
 *                   minus the frames of earlier calls); -1 where a row had
 *                   already finished.
 *   frames_emitted  [batch] int32 host or NULL: total frames per row so far
 *   finish_reason   [batch] int32 host or NULL: Q3_RUNNING / Q3_FINISHED_*
 * Consecutive calls continue exactly (a run split into calls gives the same
 * codes as one call).  Errors: Q3_ERR_STATE (no prefill), Q3_ERR_ARG,
 * Q3_ERR_NAN (a row's logits held NaN/+inf: that row ends with
 * Q3_FINISHED_ERROR, the others continue), Q3_ERR_BOUNDS, Q3_ERR_CUDA. */
int q3tts_step_frames(q3tts_t* h, int n_frames, int32_t* codes_out, int32_t* frames_emitted,
                      int32_t* finish_reason);

/* Talker-width rows of text tokens ("Qwen3-TTS 移植 ncnn 简明教程" section 1,
 * talker bullet: Qwen2 BPE ids -> 2048-d text embedding -> ResizeMLP
 * (2048 -> 2048 -> talker width, SiLU); the trailing-text rows that q3tts_prefill
 * takes, one consumed per talker step):
 *   rows_out[i] = fc2_w . silu(fc1_w . text_emb[ids[i]] + fc1_b) + fc2_b
 * Every step runs on the GPU (an embedding gather, then the two projections
 * as tensor-core GEMMs from 16 ids on, GEMVs below).
 *   n         ids, >= 0
 *   ids       [n] int32, host or device, each in [0, text_vocab)
 *   rows_out  [n][hidden] f32, host or device
 * Errors: Q3_ERR_ARG (no text path in the config or weights, NULL pointer, a
 * host id out of range), Q3_ERR_BOUNDS (a device id out of range; its row is
 * left zero), Q3_ERR_CUDA.  Ends with one synchronisation of the stream. */
int q3tts_text_embed(q3tts_t* h, int n, const int32_t* ids, float* rows_out);

/* Parity capture: while set, every talker selection of the listed rows stores
 * its raw fp32 logits to talker_logits[slot][k][codec_vocab] (k = selection
 * index, 0..max_frames) and every predictor draw stores to
 * cp_logits[slot][f][n_groups-1][cp_vocab] (f = frame).  Device pointers,
 * borrowed until the capture is cleared (n_rows = 0) or the handle destroyed.
 * max_frames bounds k and f; selections beyond it are not stored.  */
int q3tts_set_capture(q3tts_t* h, int n_rows, const int32_t* rows, float* talker_logits, float* cp_logits,
                      int max_frames);

/* The logits processors and draw on caller-given logits, for testing the
 * sampler bit for bit (same kernel as the frame loop).  The chain and its
 * order: repetition penalty over the row's drawn ids, EOS masked while
 * k < min_new_tokens, suppression of [suppress_lo, suppress_hi) except EOS,
 * then greedy or temperature -> top-k -> top-p -> argmax(p / Exp(1))
 * (ncnn discussion 6832 §3.2 logits processors; "Qwen3-TTS 移植 ncnn 简明教程"
 * §1 fact 3 and §6 processor order; Mizuoto page 速度 for the draw).
 *   n               logit sets
 *   logits          [n][V] f32 device; V = codec_vocab if talker else cp_vocab
 *   talker          1: talker chain (penalty, min_new, suppression) then draw;
 *                   0: predictor draw (cp_* settings)
 *   params          [n] host: settings of each set
 *   seen            [n][V] uint8 device or NULL: ids already selected (penalty)
 *   sel_index       [n] host: selection index k (min_new_tokens) and frame
 *                   index of the noise counter
 *   step            noise step (0 talker, q = 1..15 predictor codebook)
 *   noise_row       [n] host: row index of the noise counter
 *   ids_out         [n] int32 host
 * Errors: Q3_ERR_NAN (ids_out of a NaN set is -1), Q3_ERR_ARG (also: a set
 * that samples with temperature <= 0, or a talker set with repetition_penalty
 * <= 0; nothing is run), Q3_ERR_CUDA. */
int q3tts_sample_logits(q3tts_t* h, int n, const float* logits, int talker, const q3tts_sampling* params,
                        const uint8_t* seen, const int32_t* sel_index, int step, const int32_t* noise_row,
                        int32_t* ids_out);

/* The logits processors and draw of q3tts_sample_logits, for callers that
 * cannot allocate device memory (no handle, no workspace): e.g. code running
 * inside another allocator's callback, a real-time thread that must never
 * block on an allocator, or a process whose device memory is fully reserved
 * by another runtime.  The pages have no counterpart of this entry point.
 *   n               logit sets, 0..1024 (more: Q3_ERR_CAPACITY, nothing done)
 *   vocab           entries per set (2..4096)
 *   logits          [n][vocab] f32, DEVICE memory
 *   talker, params, sel_index, step, noise_row: as in q3tts_sample_logits
 *                   (params / sel_index / noise_row are host arrays)
 *   seen            [n][vocab] uint8 DEVICE memory or NULL
 *   eos_id, suppress_lo, suppress_hi: the talker chain's specials
 *   ids_out         [n] int32 HOST memory (-1 for a NaN set)
 *   stream          cudaStream_t (NULL = legacy default stream); the call
 *                   ends with one synchronisation of it
 * Staging lives in a fixed device array (about 70 KB per GPU that loads the
 * library, kept until the process exits); the library calls no allocator.
 * The first call on each device looks the array's address up, so make that
 * first call before any stream capture.  Every call reuses the same array:
 * calls that overlap on the GPU (other streams, other threads) race and must
 * be serialised by the caller.  Errors: Q3_ERR_CAPACITY, Q3_ERR_ARG (as in
 * q3tts_sample_logits, including the per-set settings), Q3_ERR_NAN,
 * Q3_ERR_CUDA. */
int q3tts_sample_logits_noalloc(int n, int vocab, const float* logits, int talker, const q3tts_sampling* params,
                                const uint8_t* seen, const int32_t* sel_index, int step, const int32_t* noise_row,
                                int eos_id, int suppress_lo, int suppress_hi, int32_t* ids_out, void* stream);

/* Number of kernel launches one talker step of the current batch makes (the
 * kernel nodes of the step's CUDA graph, which this call records if needed).
 * Errors: Q3_ERR_STATE (no prefill), Q3_ERR_CUDA. */
int q3tts_step_kernel_count(q3tts_t* h, int* count);

/* The path that runs one talker step of a batch of `batch` rows on this
 * handle: Q3_PATH_CLUSTER, Q3_PATH_FRAME (batch 1 only) or Q3_PATH_GRAPH.
 * Errors: Q3_ERR_ARG (NULL pointer, batch outside 1..max_batch). */
int q3tts_step_path(const q3tts_t* h, int batch, int* path);

/* One-line description of the last error on this handle. */
const char* q3tts_last_error(const q3tts_t* h);

/* Release the handle (not the borrowed weights or workspace). */
void q3tts_destroy(q3tts_t* h);

#ifdef __cplusplus
}
#endif
#endif /* Q3TTS_H */
