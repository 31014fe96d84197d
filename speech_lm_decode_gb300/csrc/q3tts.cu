// Host side of the C ABI in q3tts.h: validation, workspace layout, the
// prefill, and the per-step kernel sequence recorded once as a CUDA graph and
// replayed for every talker step (one host synchronisation per call).
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "cluster_step.h"
#include "frame_params.h"
#include "kernels.h"

using namespace q3;

namespace {

constexpr size_t ALIGN = 256;
constexpr int PREFILL_CHUNK = 8192;  // prompt tokens per prefill pass (enough token tiles to fill the GPU)
constexpr int MAX_SPLITS = 16;       // split-KV partitions per (token, kv head)
constexpr int MIN_SAMPLE_SETS = 256; // staging for q3tts_sample_logits

struct Layout {
    size_t kvK, kvV, ckvK, ckvV, rope, rows, params, h, x, cx, tok, opA, opB, headop, qkv, pm, pl, pacc, logits,
        cplogits, t_row, t_pos, c_row, c_pos, last_row, codes, codes_stage, text, pad, err, s_params, s_logits, s_sel, s_row, s_ids, s_seen, cap_slot,
        fparams, fctl, fpart, fll, tcs, tcs2, clpack, clxr, cllg, clparams, ptiles;
    bool cl;                            // the cluster step kernel's regions are present
    size_t total;
    int mmax, kA, kB, rope_rows, frames_cap, n_sets, vmax, fsplits;
    size_t fll_words;                   // exchange words of the frame kernel
    size_t fw_x, fw_cx, fw_qkv, fw_o, fw_act, fw_log, fw_cpl;   // word offsets in fll
};

size_t esize(int dtype) { return dtype == Q3_BF16 ? 2 : 4; }

Layout make_layout(const q3tts_config& c) {
    Layout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off += (bytes + ALIGN - 1) / ALIGN * ALIGN;
        return o;
    };
    const size_t e = esize(c.dtype);
    const size_t B = (size_t)c.max_batch, hd = (size_t)c.head_dim;
    const int nqkv = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
    L.mmax = std::max(std::min(PREFILL_CHUNK, c.max_batch * c.max_ctx), 2 * c.max_batch);
    L.kA = std::max(std::max(std::max(c.hidden, c.cp_hidden), c.n_q_heads * c.head_dim), c.text_hidden);
    L.kB = std::max(std::max(std::max(c.ffn, c.cp_ffn), c.hidden), c.text_hidden);
    L.rope_rows = std::max(c.max_ctx, 16);
    L.frames_cap = c.max_ctx;
    L.n_sets = std::max(c.max_batch, MIN_SAMPLE_SETS);
    L.vmax = std::max(c.codec_vocab, c.cp_vocab);
    const size_t kv = (size_t)c.n_layers * B * c.n_kv_heads * c.max_ctx * hd * e;
    L.kvK = take(kv);
    L.kvV = take(kv);
    const size_t ckv = (size_t)c.cp_layers * B * c.n_kv_heads * 16 * hd * e;
    L.ckvK = take(ckv);
    L.ckvV = take(ckv);
    L.rope = take((size_t)L.rope_rows * (hd / 2) * 2 * sizeof(float));
    L.rows = take(B * sizeof(RowState));
    L.params = take(B * sizeof(q3tts_sampling));
    L.h = take(B * c.hidden * sizeof(float));
    L.x = take((size_t)L.mmax * c.hidden * sizeof(float));
    L.cx = take(2 * B * c.cp_hidden * sizeof(float));
    L.tok = take(2 * B * c.hidden * sizeof(float));
    L.opA = take((size_t)L.mmax * L.kA * sizeof(float));
    L.opB = take((size_t)L.mmax * L.kB * sizeof(float));
    L.headop = take(B * c.hidden * sizeof(float));
    L.qkv = take((size_t)L.mmax * nqkv * sizeof(float));
    // split-KV partials: up to MAX_SPLITS splits for decode batches (<= 2B tokens),
    // one split for longer prefill chunks
    const size_t np = std::max((size_t)L.mmax, 2 * B * MAX_SPLITS) * c.n_q_heads;
    L.pm = take(np * sizeof(float));
    L.pl = take(np * sizeof(float));
    L.pacc = take(np * hd * sizeof(float));
    L.logits = take(B * c.codec_vocab * sizeof(float));
    L.cplogits = take(B * c.cp_vocab * sizeof(float));
    L.t_row = take((size_t)L.mmax * sizeof(int));
    L.t_pos = take((size_t)L.mmax * sizeof(int));
    L.c_row = take((size_t)MAX_GROUPS * 2 * B * sizeof(int));
    L.c_pos = take((size_t)MAX_GROUPS * 2 * B * sizeof(int));
    L.last_row = take((size_t)L.mmax * sizeof(int));
    L.ptiles = take((size_t)L.mmax * 4 * sizeof(int));   // prefill attention tiles of one chunk
    L.codes = take(B * L.frames_cap * MAX_GROUPS * sizeof(int32_t));
    L.codes_stage = take(B * L.frames_cap * MAX_GROUPS * sizeof(int32_t));
    L.text = take(B * std::max(c.max_text, 1) * c.hidden * sizeof(float));
    L.pad = take(c.hidden * sizeof(float));
    L.err = take(4 * sizeof(int));
    L.s_params = take((size_t)L.n_sets * sizeof(q3tts_sampling));
    L.s_logits = take((size_t)L.n_sets * L.vmax * sizeof(float));
    L.s_sel = take((size_t)L.n_sets * sizeof(int));
    L.s_row = take((size_t)L.n_sets * sizeof(int));
    L.s_ids = take((size_t)L.n_sets * sizeof(int));
    L.s_seen = take((size_t)L.n_sets * L.vmax);
    L.cap_slot = take(B * sizeof(int));
    // persistent frame kernel (batch 1)
    L.fsplits = 16;   // partial buffers sized for the largest split count
    L.fparams = take(sizeof(FrameParams));
    L.fctl = take(FRAME_CTL_WORDS * sizeof(unsigned));
    L.fpart = take((size_t)c.n_kv_heads * L.fsplits * (c.n_q_heads / c.n_kv_heads) * (HD + 2) * sizeof(float));
    {
        size_t w = 0;
        auto words = [&](size_t n) { size_t o = w; w += (n + 31) / 32 * 32; return o; };
        L.fw_x = words(c.hidden);
        L.fw_cx = words(2 * (size_t)c.cp_hidden);
        L.fw_qkv = words(2 * (size_t)nqkv);
        L.fw_o = words(2 * (size_t)c.n_q_heads * HD);
        L.fw_act = words(2 * (size_t)std::max(c.ffn, c.cp_ffn));
        L.fw_log = words(c.codec_vocab);
        L.fw_cpl = words(c.cp_vocab);
        L.fll_words = w;
        L.fll = take(w * sizeof(Word));
    }
    // tensor-core path: bf16 high / low parts of an fp32 operand [mmax][kmax]
    L.tcs = c.dtype == Q3_BF16 ? take((size_t)L.mmax * std::max(L.kA, L.kB) * 4) : take(256);
    // a second one: the SiLU(g)*u operand of the down projection, written while the
    // gate/up projection still reads the first
    // (also the up product's fp32 output [mmax][F] when q/k/v and gate/up run
    // as separate products)
    L.tcs2 = c.dtype == Q3_BF16 || c.separate_projections ? take((size_t)L.mmax * std::max(L.kA, L.kB) * 4)
                                                          : take(256);
    // cluster step kernel (batch 1): packed weight image, exchange words, parameters
    L.cl = c.step_path == Q3_PATH_CLUSTER && cl_unsupported(c)[0] == 0;
    if (L.cl) {
        const ClLayout cl = cl_layout(c);
        L.clpack = take(cl.pack_bytes);
        L.clxr = take(cl.xr_words * sizeof(Word));
        L.cllg = take(cl.lg_words * sizeof(Word));
        L.clparams = take(sizeof(ClParams));
    }
    L.total = off;
    return L;
}

bool config_ok(const q3tts_config* c, std::string* why) {
    auto bad = [&](const char* m) { if (why) *why = m; return false; };
    if (!c) return bad("config is NULL");
    if (c->head_dim != HD) return bad("head_dim must be 128");
    if (c->n_layers < 1 || c->cp_layers < 1) return bad("layer counts must be >= 1");
    if (c->n_kv_heads < 1 || c->n_q_heads % c->n_kv_heads) return bad("n_q_heads must be a multiple of n_kv_heads");
    const int g = c->n_q_heads / c->n_kv_heads;
    if (g != 1 && g != 2 && g != 4) return bad("n_q_heads / n_kv_heads must be 1, 2 or 4");
    if (c->n_q_heads + c->n_kv_heads > 32) return bad("n_q_heads + n_kv_heads must be <= 32");
    for (int v : {c->hidden, c->ffn, c->cp_hidden, c->cp_ffn})
        if (v < 8 || v % 8) return bad("hidden / ffn widths must be positive multiples of 8");
    if (c->n_groups < 2 || c->n_groups > MAX_GROUPS) return bad("n_groups must be in [2, 16]");
    if (c->codec_vocab < 2 || c->codec_vocab > MAX_VOCAB || c->cp_vocab < 2 || c->cp_vocab > MAX_VOCAB)
        return bad("vocabularies must be in [2, 4096]");
    if (c->eos_id < 0 || c->eos_id >= c->codec_vocab) return bad("eos_id out of range");
    if (c->suppress_lo < 0 || c->suppress_hi > c->codec_vocab || c->suppress_lo > c->suppress_hi)
        return bad("suppress range out of range");
    if (c->dtype != Q3_F32 && c->dtype != Q3_BF16) return bad("dtype must be Q3_F32 or Q3_BF16");
    if (c->max_batch < 1 || c->max_ctx < 2 || c->max_text < 0) return bad("bad max_batch / max_ctx / max_text");
    if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) return bad("bad rms_eps / rope_theta");
    if (c->step_path < Q3_PATH_AUTO || c->step_path > Q3_PATH_CLUSTER) return bad("step_path out of range");
    if (c->wait_limit_us < 0 || c->inject_timeout < 0 || c->debug_sync < 0 || c->debug_sync > 1)
        return bad("bad wait_limit_us / inject_timeout / debug_sync");
    if (c->separate_projections < 0 || c->separate_projections > 1) return bad("separate_projections must be 0 or 1");
    if (c->step_path == Q3_PATH_CLUSTER && cl_unsupported(*c)[0] != 0) return bad("cluster kernel: unsupported shape");
    if (c->text_vocab < 0 || c->text_hidden < 0 || (c->text_vocab > 0) != (c->text_hidden > 0) ||
        (c->text_hidden > 0 && c->text_hidden % 8))
        return bad("text_vocab / text_hidden: both 0, or both positive with text_hidden a multiple of 8");
    return true;
}

template <typename T>
T* at(void* base, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(base) + off); }

}  // namespace

struct q3tts {
    q3tts_config c;
    q3tts_weights w;
    Layout L;
    void* ws = nullptr;
    cudaStream_t st = nullptr;
    bool own_stream = false;
    std::string last_error;
    int batch = 0;
    bool prefilled = false;
    long steps_done = 0;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    int graph_batch = -1;
    float* cap_t = nullptr;
    float* cap_c = nullptr;
    int cap_T = 0;
    bool capturing = false;
    int splits_t = 1;
    bool cl_ok = false;         // the cluster step kernel serves batch 1
    bool frame_ok = false;      // the persistent frame kernel can serve batch 1
    bool frame_tc = false;      // ... with its GEMV rows on the tensor cores
    size_t frame_smem = 0;
    int frame_grid = 0;
    int frame_xin = 0;
    int frame_splits = 1;

    template <typename T> T* p(size_t off) const { return at<T>(ws, off); }
    TcScratch tc() const {
        TcScratch t;
        t.base = c.dtype == Q3_BF16 ? p<void>(L.tcs) : nullptr;
        t.bytes = c.dtype == Q3_BF16 ? (size_t)L.mmax * std::max(L.kA, L.kB) * 4 : 0;
        t.min_tokens = c.tc_min_tokens == 0 ? 16 : c.tc_min_tokens;
        return t;
    }
    TcScratch tc2() const {
        TcScratch t = tc();
        t.base = c.dtype == Q3_BF16 ? p<void>(L.tcs2) : nullptr;
        return t;
    }
    RowState* rows() const { return p<RowState>(L.rows); }
    int* err() const { return p<int>(L.err); }
};

namespace {

int fail(q3tts* h, int code, const char* fmt, ...) {
    if (h) {
        char buf[512];
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(buf, sizeof buf, fmt, ap);
        va_end(ap);
        h->last_error = buf;
    }
    return code;
}

#define CK(call)                                                                                    \
    do {                                                                                            \
        cudaError_t e_ = (call);                                                                    \
        if (e_ != cudaSuccess) return fail(h, Q3_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
    } while (0)

// Opt-in launch-by-launch check (config debug_sync = 1): outside graph
// capture, wait up to 20 s for each launch, report it on stderr, and end the
// process if it did not finish (the driver then tears the context down).
void debug_wait(const q3tts* h, const char* what) {
    if (!h->c.debug_sync) return;
    cudaStream_t st = h->st;
    cudaStreamCaptureStatus cs;
    if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone) return;
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        const cudaError_t e = cudaStreamQuery(st);
        const double dt = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
        if (e == cudaSuccess) { fprintf(stderr, "[q3tts] ok %.3f ms  %s\n", dt * 1e3, what); return; }
        if (e != cudaErrorNotReady) { fprintf(stderr, "[q3tts] error %s after %s\n", cudaGetErrorString(e), what); return; }
        if (dt > 20.0) { fprintf(stderr, "[q3tts] DID NOT FINISH in 20 s: %s\n", what); fflush(stderr); std::_Exit(3); }
    }
}

// NVTX range for profilers (header-only NVTX3; no cost without a tool attached)
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

void invalidate_graph(q3tts* h) {
    if (h->exec) cudaGraphExecDestroy(h->exec);
    if (h->graph) cudaGraphDestroy(h->graph);
    h->exec = nullptr;
    h->graph = nullptr;
    h->graph_batch = -1;
}

// One decoder stack over M tokens (talker or predictor), residual x [M][H].
// tiles / n_tiles: prompt tokens of a prefill chunk, whose attention runs tiled
// (bf16 caches); NULL for decode steps.  single: every token belongs to a
// different row (a decode step), so short bf16 caches take the attention with
// QK-norm, RoPE and the cache append fused in.
int enqueue_layers(q3tts* h, bool talker, int M, float* x, const int* trow, const int* tpos,
                   const int4* tiles = nullptr, int n_tiles = 0, bool single = false) {
    const q3tts_config& c = h->c;
    const q3tts_block_weights& bw = talker ? h->w.talker : h->w.cp;
    const int L = talker ? c.n_layers : c.cp_layers;
    const int H = talker ? c.hidden : c.cp_hidden;
    const int F = talker ? c.ffn : c.cp_ffn;
    const int cap = talker ? c.max_ctx : 16;
    const int nq = c.n_q_heads, nkv = c.n_kv_heads, hd = c.head_dim;
    const int nqkv = (nq + 2 * nkv) * hd;
    const size_t e = esize(c.dtype);
    const size_t kv_layer = (size_t)c.max_batch * nkv * cap * hd * e;
    char* Kc = h->p<char>(talker ? h->L.kvK : h->L.ckvK);
    char* Vc = h->p<char>(talker ? h->L.kvV : h->L.ckvV);
    float* opA = h->p<float>(h->L.opA);
    float* opB = h->p<float>(h->L.opB);
    float* qkv = h->p<float>(h->L.qkv);
    const int splits = talker ? (M <= 2 * c.max_batch ? h->splits_t : 1) : 1;
    const float eps = c.rms_eps;
    const bool presplit = linear_takes_split(c.dtype, M, H, h->tc());
    // the attention combine writes the O projection's operand, and the gate/up
    // projection the down projection's, when those run on the tensor cores
    const TcScratch tcs = h->tc(), tcs2 = h->tc2();
    const bool presplit_o = linear_takes_split(c.dtype, M, c.n_q_heads * c.head_dim, tcs);
    const bool presplit_d = presplit && linear_takes_split(c.dtype, M, F, tcs2);
    for (int l = 0; l < L; ++l) {
        const char* wqkv = (const char*)bw.wqkv + (size_t)l * nqkv * H * e;
        const char* wo = (const char*)bw.wo + (size_t)l * H * nq * hd * e;
        const char* wgu = (const char*)bw.wgu + (size_t)l * 2 * F * H * e;
        const char* wd = (const char*)bw.wd + (size_t)l * H * F * e;
        // RMSNorm + q/k/v projection (the norm writes the tensor-core operand directly when that path runs)
        if (presplit) {
            CK(launch_rmsnorm_split(x, H, M, (const float*)bw.attn_norm + (size_t)l * H, H, eps, h->tc(), h->st)); debug_wait(h, "launch_rmsnorm_split");
        } else {
            CK(launch_rmsnorm(x, H, M, (const float*)bw.attn_norm + (size_t)l * H, H, eps, opA, H, nullptr, 0,
                              nullptr, h->st)); debug_wait(h, "launch_rmsnorm");
        }
        if (c.separate_projections) {
            // q, k and v rows as three products into their columns of qkv
            const int part[4] = {0, nq * hd, (nq + nkv) * hd, nqkv};
            for (int i = 0; i < 3; ++i) {
                CK(launch_linear(c.dtype, wqkv + (size_t)part[i] * H * e, part[i + 1] - part[i], H,
                                 presplit ? nullptr : opA, H, M, qkv + part[i], nqkv, nullptr, 0, h->tc(), h->err(),
                                 h->st)); debug_wait(h, "launch_linear");
            }
        } else {
            CK(launch_linear(c.dtype, wqkv, nqkv, H, presplit ? nullptr : opA, H, M, qkv, nqkv, nullptr, 0, h->tc(), h->err(), h->st)); debug_wait(h, "launch_linear");
        }
        const bool fused = single && !tiles && c.dtype == Q3_BF16 && nq == 2 * nkv && cap <= 64;
        if (fused) {
            CK(launch_attention_short_fused(qkv, nqkv, M, nq, nkv, (const float*)bw.q_norm + (size_t)l * hd,
                                            (const float*)bw.k_norm + (size_t)l * hd, eps, h->p<float>(h->L.rope),
                                            h->L.rope_rows, Kc + l * kv_layer, Vc + l * kv_layer, cap, trow, tpos, opA,
                                            nq * hd, h->err(), h->st, presplit_o ? &tcs : nullptr));
            debug_wait(h, "launch_attention_short_fused");
        } else {
            CK(launch_qk_rope_kv(c.dtype, qkv, nqkv, M, nq, nkv, (const float*)bw.q_norm + (size_t)l * hd,
                                 (const float*)bw.k_norm + (size_t)l * hd, eps, h->p<float>(h->L.rope),
                                 h->L.rope_rows, Kc + l * kv_layer, Vc + l * kv_layer, cap, trow, tpos, h->err(),
                                 h->st)); debug_wait(h, "launch_qk_rope_kv");
        }
        if (!fused && tiles && c.dtype == Q3_BF16) {
            CK(launch_prefill_attention(c.dtype, qkv, nqkv, M, nq, nkv, Kc + l * kv_layer, Vc + l * kv_layer, cap,
                                        tiles, n_tiles, opA, nq * hd, h->st, presplit_o ? &tcs : nullptr));
            debug_wait(h, "launch_prefill_attention");
        } else if (!fused) {
            CK(launch_attention(c.dtype, qkv, nqkv, M, nq, nkv, Kc + l * kv_layer, Vc + l * kv_layer, cap, trow, tpos,
                                splits, h->p<float>(h->L.pm), h->p<float>(h->L.pl), h->p<float>(h->L.pacc), opA,
                                nq * hd, h->err(), h->st, presplit_o ? &tcs : nullptr));
            debug_wait(h, "launch_attention");
        }
        CK(launch_linear(c.dtype, wo, H, nq * hd, presplit_o ? nullptr : opA, nq * hd, M, x, H, nullptr, 1, tcs, h->err(),
                         h->st)); debug_wait(h, "launch_linear");
        if (presplit) {
            CK(launch_rmsnorm_split(x, H, M, (const float*)bw.mlp_norm + (size_t)l * H, H, eps, h->tc(), h->st)); debug_wait(h, "launch_rmsnorm_split");
        } else {
            CK(launch_rmsnorm(x, H, M, (const float*)bw.mlp_norm + (size_t)l * H, H, eps, opA, H, nullptr, 0,
                              nullptr, h->st)); debug_wait(h, "launch_rmsnorm");
        }
        if (c.separate_projections) {
            // gate into opB, up into the second scratch (as fp32 [M][F]), then
            // SiLU(g) * u in place: the down projection reads opB
            float* up = h->p<float>(h->L.tcs2);
            CK(launch_linear(c.dtype, wgu, F, H, presplit ? nullptr : opA, H, M, opB, F, nullptr, 0, tcs, h->err(),
                             h->st)); debug_wait(h, "launch_linear");
            CK(launch_linear(c.dtype, wgu + (size_t)F * H * e, F, H, presplit ? nullptr : opA, H, M, up, F, nullptr,
                             0, tcs, h->err(), h->st)); debug_wait(h, "launch_linear");
            CK(launch_silu_mul(opB, up, (long)M * F, h->st)); debug_wait(h, "launch_silu_mul");
            CK(launch_linear(c.dtype, wd, H, F, opB, F, M, x, H, nullptr, 1, tcs, h->err(), h->st));
            debug_wait(h, "launch_linear");
        } else {
            CK(launch_linear_gated(c.dtype, wgu, F, H, presplit ? nullptr : opA, H, M, opB, F, tcs, h->err(), h->st,
                                   presplit_d ? &tcs2 : nullptr)); debug_wait(h, "launch_linear_gated");
            CK(launch_linear(c.dtype, wd, H, F, presplit_d ? nullptr : opB, F, M, x, H, nullptr, 1,
                             presplit_d ? tcs2 : tcs, h->err(), h->st)); debug_wait(h, "launch_linear");
        }
    }
    return Q3_OK;
}

// Predictor tokens (talker width, in h->tok) -> predictor residual cx.
int enqueue_cp_input(q3tts* h, int M) {
    const q3tts_config& c = h->c;
    if (c.hidden == c.cp_hidden) return Q3_OK;  // tokens were written to cx directly
    CK(launch_linear(c.dtype, h->w.cp_proj_w, c.cp_hidden, c.hidden, h->p<float>(h->L.tok), c.hidden, M,
                     h->p<float>(h->L.cx), c.cp_hidden, (const float*)h->w.cp_proj_b, 0, h->tc(), h->err(), h->st)); debug_wait(h, "launch_linear");
    return Q3_OK;
}

// One talker step for the whole batch: complete frame k-1 through the code
// predictor, assemble the next talker input, run the talker, select code0.
int enqueue_frame(q3tts* h) {
    CK(launch_frame(h->c.dtype, h->frame_tc, h->p<FrameParams>(h->L.fparams), h->frame_grid, h->frame_smem, h->st)); debug_wait(h, "launch_frame");
    return Q3_OK;
}

int enqueue_step(q3tts* h) {
    if (h->batch == 1 && h->cl_ok) {
        CK(launch_cluster_step(h->p<ClParams>(h->L.clparams), h->st)); debug_wait(h, "launch_cluster_step");
        return Q3_OK;
    }
    if (h->batch == 1 && h->frame_ok) return enqueue_frame(h);
    const q3tts_config& c = h->c;
    const int B = h->batch, G1 = c.n_groups - 1;
    const size_t e = esize(c.dtype);
    RowState* rs = h->rows();
    const q3tts_sampling* P = h->p<q3tts_sampling>(h->L.params);
    int* t_row = h->p<int>(h->L.t_row);
    int* t_pos = h->p<int>(h->L.t_pos);
    int* c_row = h->p<int>(h->L.c_row);
    int* c_pos = h->p<int>(h->L.c_pos);
    int32_t* codes = h->p<int32_t>(h->L.codes);
    float* cx = h->p<float>(h->L.cx);
    float* tok = (c.hidden == c.cp_hidden) ? cx : h->p<float>(h->L.tok);
    float* opA = h->p<float>(h->L.opA);
    float* cpl = h->p<float>(h->L.cplogits);
    const int* slot = h->p<int>(h->L.cap_slot);
    int r;

    CK(launch_prepare_step(rs, B, t_row, t_pos, c_row, c_pos, G1, h->st)); debug_wait(h, "launch_prepare_step");
    // code predictor: 2-token prefill -> head[0] -> codebook 1
    CK(launch_cp_embed_prefill(c.dtype, rs, B, h->p<float>(h->L.h), h->w.codec_emb, c.hidden, c.codec_vocab, codes,
                               h->L.frames_cap, tok, h->err(), h->st)); debug_wait(h, "launch_cp_embed_prefill");
    if ((r = enqueue_cp_input(h, 2 * B))) return r;
    if ((r = enqueue_layers(h, false, 2 * B, cx, c_row, c_pos))) return r;
    CK(launch_rmsnorm(cx + c.cp_hidden, 2 * c.cp_hidden, B, (const float*)h->w.cp.final_norm, c.cp_hidden,
                      c.rms_eps, opA, c.cp_hidden, nullptr, 0, nullptr, h->st)); debug_wait(h, "launch_rmsnorm");
    CK(launch_linear(c.dtype, h->w.cp_heads, c.cp_vocab, c.cp_hidden, opA, c.cp_hidden, B, cpl, c.cp_vocab, nullptr,
                     0, h->tc(), h->err(), h->st)); debug_wait(h, "launch_linear");
    CK(launch_cp_sample(cpl, c.cp_vocab, B, rs, P, 0, codes, h->L.frames_cap, h->err(), h->cap_c, slot, h->cap_T,
                        c.n_groups, h->st)); debug_wait(h, "launch_cp_sample");
    // 14 autoregressive steps: table[s-1](code s) at position s+1 -> head[s] -> codebook s+1
    for (int s = 1; s < G1; ++s) {
        CK(launch_cp_embed_step(c.dtype, rs, B, h->w.cp_emb, c.hidden, c.cp_vocab, s, codes, h->L.frames_cap, tok,
                                h->err(), h->st)); debug_wait(h, "launch_cp_embed_step");
        if ((r = enqueue_cp_input(h, B))) return r;
        if ((r = enqueue_layers(h, false, B, cx, c_row + (size_t)s * 2 * B, c_pos + (size_t)s * 2 * B, nullptr, 0,
                                true))) return r;
        CK(launch_rmsnorm(cx, c.cp_hidden, B, (const float*)h->w.cp.final_norm, c.cp_hidden, c.rms_eps, opA,
                          c.cp_hidden, nullptr, 0, nullptr, h->st)); debug_wait(h, "launch_rmsnorm");
        const char* head = (const char*)h->w.cp_heads + (size_t)s * c.cp_vocab * c.cp_hidden * e;
        CK(launch_linear(c.dtype, head, c.cp_vocab, c.cp_hidden, opA, c.cp_hidden, B, cpl, c.cp_vocab, nullptr, 0,
                         h->tc(), h->err(), h->st)); debug_wait(h, "launch_linear");
        CK(launch_cp_sample(cpl, c.cp_vocab, B, rs, P, s, codes, h->L.frames_cap, h->err(), h->cap_c, slot, h->cap_T,
                            c.n_groups, h->st)); debug_wait(h, "launch_cp_sample");
    }
    // talker step
    float* x = h->p<float>(h->L.x);
    CK(launch_talker_embed(c.dtype, rs, B, h->w.codec_emb, h->w.cp_emb, c.hidden, c.codec_vocab, c.cp_vocab,
                           c.n_groups, codes, h->L.frames_cap, h->p<float>(h->L.text), h->p<float>(h->L.pad), x,
                           c.eos_id, h->err(), h->st)); debug_wait(h, "launch_talker_embed");
    if ((r = enqueue_layers(h, true, B, x, t_row, t_pos, nullptr, 0, true))) return r;
    CK(launch_rmsnorm(x, c.hidden, B, (const float*)h->w.talker.final_norm, c.hidden, c.rms_eps, opA,
                      c.hidden, h->p<float>(h->L.h), c.hidden, nullptr, h->st)); debug_wait(h, "launch_rmsnorm");
    float* logits = h->p<float>(h->L.logits);
    CK(launch_linear(c.dtype, h->w.codec_head, c.codec_vocab, c.hidden, opA, c.hidden, B, logits, c.codec_vocab,
                     nullptr, 0, h->tc(), h->err(), h->st)); debug_wait(h, "launch_linear");
    CK(launch_talker_sample(logits, c.codec_vocab, B, rs, P, c.eos_id, c.suppress_lo, c.suppress_hi, 1, h->err(),
                            h->cap_t, slot, h->cap_T, h->st)); debug_wait(h, "launch_talker_sample");
    return Q3_OK;
}

// Record one talker step of the current batch as a CUDA graph.
int record_step_graph(q3tts* h) {
    CK(cudaStreamBeginCapture(h->st, cudaStreamCaptureModeThreadLocal));
    int r = enqueue_step(h);
    cudaGraph_t g = nullptr;
    cudaError_t e = cudaStreamEndCapture(h->st, &g);
    if (r) { if (g) cudaGraphDestroy(g); return r; }
    if (e != cudaSuccess) return fail(h, Q3_ERR_CUDA, "graph capture: %s", cudaGetErrorString(e));
    h->graph = g;
    e = cudaGraphInstantiate(&h->exec, g, 0);
    if (e != cudaSuccess) {
        invalidate_graph(h);
        return fail(h, Q3_ERR_CUDA, "graph instantiate: %s", cudaGetErrorString(e));
    }
    h->graph_batch = h->batch;
    return Q3_OK;
}

// Parameters of the cluster step kernel (device copy in the workspace).
int upload_cluster_params(q3tts* h) {
    const q3tts_config& c = h->c;
    ClParams P{};
    P.pack = h->p<unsigned char>(h->L.clpack);
    P.lay = cl_layout(c);
    const q3tts_block_weights& t = h->w.talker;
    const q3tts_block_weights& k = h->w.cp;
    P.t_attn_norm = (const float*)t.attn_norm; P.t_q_norm = (const float*)t.q_norm; P.t_k_norm = (const float*)t.k_norm;
    P.t_mlp_norm = (const float*)t.mlp_norm; P.t_final_norm = (const float*)t.final_norm;
    P.c_attn_norm = (const float*)k.attn_norm; P.c_q_norm = (const float*)k.q_norm; P.c_k_norm = (const float*)k.k_norm;
    P.c_mlp_norm = (const float*)k.mlp_norm; P.c_final_norm = (const float*)k.final_norm;
    P.codec_emb = h->w.codec_emb; P.cp_emb = h->w.cp_emb; P.cp_proj_b = (const float*)h->w.cp_proj_b;
    P.H = c.hidden; P.Hc = c.cp_hidden; P.F = c.ffn; P.Fc = c.cp_ffn; P.Lt = c.n_layers; P.Lc = c.cp_layers;
    P.V = c.codec_vocab; P.cpV = c.cp_vocab; P.G = c.n_groups; P.eos = c.eos_id; P.sup_lo = c.suppress_lo;
    P.sup_hi = c.suppress_hi; P.max_batch = c.max_batch; P.cap = c.max_ctx;
    P.eps = c.rms_eps;
    P.rope = h->p<float2>(h->L.rope);
    P.Kc = h->p<void>(h->L.kvK); P.Vc = h->p<void>(h->L.kvV);
    P.rows = h->rows(); P.P = h->p<q3tts_sampling>(h->L.params);
    P.xr = h->p<Word>(h->L.clxr); P.lg = h->p<Word>(h->L.cllg);
    P.h = h->p<float>(h->L.h);
    P.codes = h->p<int32_t>(h->L.codes); P.frames_cap = h->L.frames_cap;
    P.text = h->p<float>(h->L.text); P.pad = h->p<float>(h->L.pad);
    P.ctl = h->p<unsigned>(h->L.fctl); P.err = h->err();
    P.cap_t = h->cap_t; P.cap_c = h->cap_c; P.cap_slot = h->p<int>(h->L.cap_slot); P.cap_T = h->cap_T;
    P.wait_ns = (long long)(c.wait_limit_us > 0 ? c.wait_limit_us : 2000000) * 1000;
    P.inject_skip = c.inject_timeout > 0 ? c.inject_timeout : -1;
    CK(cudaMemcpyAsync(h->p<ClParams>(h->L.clparams), &P, sizeof P, cudaMemcpyHostToDevice, h->st));
    CK(cudaStreamSynchronize(h->st));
    return Q3_OK;
}

// Parameters of the persistent frame kernel (device copy in the workspace).
int upload_frame_params(q3tts* h) {
    if (h->cl_ok) {
        int r = upload_cluster_params(h);
        if (r) return r;
    }
    if (!h->frame_ok) return Q3_OK;
    const q3tts_config& c = h->c;
    FrameParams P{};
    auto blk = [&](PBlk& d, const q3tts_block_weights& w, bool talker) {
        d.attn_norm = (const float*)w.attn_norm; d.wqkv = w.wqkv; d.q_norm = (const float*)w.q_norm;
        d.k_norm = (const float*)w.k_norm; d.wo = w.wo; d.mlp_norm = (const float*)w.mlp_norm; d.wgu = w.wgu;
        d.wd = w.wd; d.final_norm = (const float*)w.final_norm;
        d.Kc = h->p<void>(talker ? h->L.kvK : h->L.ckvK);
        d.Vc = h->p<void>(talker ? h->L.kvV : h->L.ckvV);
        d.cap = talker ? c.max_ctx : 16;
        d.L = talker ? c.n_layers : c.cp_layers;
        d.H = talker ? c.hidden : c.cp_hidden;
        d.F = talker ? c.ffn : c.cp_ffn;
    };
    blk(P.t, h->w.talker, true);
    blk(P.c, h->w.cp, false);
    P.codec_emb = h->w.codec_emb; P.codec_head = h->w.codec_head; P.cp_emb = h->w.cp_emb; P.cp_heads = h->w.cp_heads;
    P.cp_proj_w = h->w.cp_proj_w; P.cp_proj_b = (const float*)h->w.cp_proj_b;
    P.H = c.hidden; P.Hc = c.cp_hidden; P.V = c.codec_vocab; P.cpV = c.cp_vocab; P.G = c.n_groups;
    P.nq = c.n_q_heads; P.nkv = c.n_kv_heads; P.eos = c.eos_id; P.sup_lo = c.suppress_lo; P.sup_hi = c.suppress_hi;
    P.n_splits = h->frame_splits;
    P.max_batch = c.max_batch;
    P.eps = c.rms_eps;
    P.rope = h->p<float2>(h->L.rope); P.rope_rows = h->L.rope_rows;
    P.rows = h->rows(); P.P = h->p<q3tts_sampling>(h->L.params);
    Word* ll = h->p<Word>(h->L.fll);
    P.x = ll + h->L.fw_x; P.cx = ll + h->L.fw_cx; P.qkv = ll + h->L.fw_qkv; P.o = ll + h->L.fw_o;
    P.act = ll + h->L.fw_act; P.logits = ll + h->L.fw_log; P.cpl = ll + h->L.fw_cpl;
    P.h = h->p<float>(h->L.h); P.part = h->p<float>(h->L.fpart);
    P.codes = h->p<int32_t>(h->L.codes); P.frames_cap = h->L.frames_cap;
    P.text = h->p<float>(h->L.text); P.pad = h->p<float>(h->L.pad);
    P.ctl = h->p<unsigned>(h->L.fctl); P.err = h->err();
    P.cap_t = h->cap_t; P.cap_c = h->cap_c; P.cap_slot = h->p<int>(h->L.cap_slot); P.cap_T = h->cap_T;
    P.xin_bytes = h->frame_xin;
    // cycles at the highest SM clock, so the wait lasts at least the limit
    P.wait_cycles = (long long)(c.wait_limit_us > 0 ? c.wait_limit_us : 2000000) * 2070;
    // test only: the readers of one phase of the first step after a prefill
    // (selection 1, epochs 1024 + phase) wait for an epoch nobody writes
    P.inject_ep = c.inject_timeout > 0 && c.inject_timeout < FRAME_MAX_PHASES ? (1u << 10) + c.inject_timeout : 0u;
    CK(cudaMemcpyAsync(h->p<FrameParams>(h->L.fparams), &P, sizeof P, cudaMemcpyHostToDevice, h->st));
    CK(cudaStreamSynchronize(h->st));
    return Q3_OK;
}

int read_errors(q3tts* h, const int* err_host) {
    if (err_host[0] & ERRB_BOUNDS) return fail(h, Q3_ERR_BOUNDS, "device bounds check failed (id or position)");
    if (err_host[0] & ERRB_NAN) return fail(h, Q3_ERR_NAN, "NaN or +inf logits at a selection");
    if (err_host[0] & ERRB_TIMEOUT) return fail(h, Q3_ERR_TIMEOUT, "a device wait timed out");
    if (err_host[0] & ERRB_LAUNCH) return fail(h, Q3_ERR_CUDA, "the cluster step kernel was not launched as 8 x 8 clusters");
    return Q3_OK;
}

bool weights_ok(const q3tts_config& c, const q3tts_weights* w) {
    if (!w) return false;
    for (const q3tts_block_weights* b : {&w->talker, &w->cp})
        if (!b->attn_norm || !b->wqkv || !b->q_norm || !b->k_norm || !b->wo || !b->mlp_norm || !b->wgu || !b->wd ||
            !b->final_norm)
            return false;
    if (!w->codec_emb || !w->codec_head || !w->cp_emb || !w->cp_heads) return false;
    if (c.hidden != c.cp_hidden && (!w->cp_proj_w || !w->cp_proj_b)) return false;
    if (c.text_vocab > 0 && (!w->text_emb || !w->text_fc1_w || !w->text_fc1_b || !w->text_fc2_w || !w->text_fc2_b))
        return false;
    return true;
}

}  // namespace

extern "C" {

size_t q3tts_workspace_bytes(const q3tts_config* cfg) {
    if (!config_ok(cfg, nullptr)) return 0;
    return make_layout(*cfg).total;
}

int q3tts_create(const q3tts_config* cfg, const q3tts_weights* w, void* workspace, size_t workspace_bytes,
                 void* stream, q3tts_t** out) {
    if (!out) return Q3_ERR_ARG;
    *out = nullptr;
    std::string why;
    if (!config_ok(cfg, &why)) return Q3_ERR_ARG;
    if (!weights_ok(*cfg, w)) return Q3_ERR_ARG;
    const Layout L = make_layout(*cfg);
    if (!workspace || workspace_bytes < L.total || ((uintptr_t)workspace % ALIGN)) return Q3_ERR_ARG;
    q3tts* h = new q3tts();
    h->c = *cfg;
    h->w = *w;
    h->L = L;
    h->ws = workspace;
    if (stream) {
        h->st = (cudaStream_t)stream;
    } else {
        if (cudaStreamCreateWithFlags(&h->st, cudaStreamNonBlocking) != cudaSuccess) { delete h; return Q3_ERR_CUDA; }
        h->own_stream = true;
    }
    if (sampler_init() != cudaSuccess) { q3tts_destroy(h); return Q3_ERR_CUDA; }
    // persistent frame kernel for batch 1: needs GQ 2, fitting shared memory and
    // one co-resident CTA per SM (cooperative launch)
    {
        int dev = 0, sms = 0, coop = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
        const int H = cfg->hidden, Hc = cfg->cp_hidden, nqh = cfg->n_q_heads * HD;
        // input-vector buffers: the widest [M][K] fp32 of any GEMV phase
        const int kx_t = std::max(std::max(H, cfg->ffn), nqh);
        const int kx_c = std::max(std::max(Hc, cfg->cp_ffn), std::max(nqh, H != Hc ? H : 0));
        h->frame_xin = (int)std::max((size_t)4 * std::max(kx_t, 2 * kx_c), frame_attn_scratch_bytes());
        const size_t e = esize(cfg->dtype);
        const bool tc_shape = cfg->dtype == Q3_BF16 && H <= 1024 && Hc <= 1024;
        const size_t tile = frame_tile_bytes(tc_shape);
        const bool tiles_fit = (size_t)H * e * 2 <= tile && (size_t)Hc * e * 2 <= tile &&
                               (size_t)std::max(cfg->ffn, cfg->cp_ffn) * e <= tile && (size_t)nqh * e <= tile;
        // tensor-core rows where the phases are short (hidden <= 1024: the chain's
        // latency dominates); FMA rows for wider models, whose phases stream
        // long weight slices and are bandwidth-bound
        h->frame_tc = tc_shape;
        h->frame_smem = frame_smem_bytes(cfg->dtype, h->frame_xin, h->frame_tc);
        const int path = cfg->step_path;
        // the cluster step kernel: shape supported, regions laid out, 8 x 8 clusters co-resident
        if (L.cl && coop && cl_setup() == cudaSuccess) {
            h->cl_ok = cl_pack_weights(*cfg, *w, h->p<unsigned char>(L.clpack), h->st) == cudaSuccess &&
                       cudaStreamSynchronize(h->st) == cudaSuccess;
        }
        cudaGetLastError();
        if (path == Q3_PATH_CLUSTER && !h->cl_ok) { q3tts_destroy(h); return Q3_ERR_ARG; }
        const bool want = path == Q3_PATH_FRAME || path == Q3_PATH_AUTO;
        h->frame_ok = want && coop && sms >= cfg->n_kv_heads && h->frame_smem > 0 && tiles_fit &&
                      cfg->cp_vocab <= FRAME_CP_VMAX &&
                      cfg->n_q_heads == 2 * cfg->n_kv_heads;
        if (h->frame_ok && frame_setup(cfg->dtype, h->frame_smem, h->frame_tc) != cudaSuccess) {
            cudaGetLastError();
            h->frame_ok = false;
        }
        if (h->frame_ok) {
            int blocks = 0;
            if (frame_occupancy(cfg->dtype, h->frame_smem, h->frame_tc, &blocks) != cudaSuccess || blocks < 1) {
                cudaGetLastError();
                h->frame_ok = false;
            }
        }
        // grid: every GEMV phase must give each CTA at least one output row (the
        // exchange words rely on it), so no more CTAs than the narrowest output
        const int nqkv = (cfg->n_q_heads + 2 * cfg->n_kv_heads) * HD;
        int grid = sms;
        for (int n : {nqkv, H, cfg->ffn, Hc, cfg->cp_ffn, cfg->codec_vocab, cfg->cp_vocab}) grid = std::min(grid, n);
        const int phases = (cfg->n_groups - 1) * ((H != Hc ? 1 : 0) + 5 * cfg->cp_layers + 2) + 5 * cfg->n_layers + 2;
        // residual rows a CTA updates in one phase fit its buffer
        auto rows = [&](int n) { return (n + grid - 1) / grid; };
        bool v_ok = rows(H) <= FRAME_MAX_ROWS && rows(Hc) <= FRAME_MAX_ROWS;
        if (cfg->dtype == Q3_BF16 && cfg->hidden <= 1024 && cfg->cp_hidden <= 1024) {
            // tensor-core rows: K in steps of 16, and a phase's partial sums (rows x
            // gate/up x vectors x 8 splits) fit the CTA's buffer
            for (int k : {H, cfg->ffn, Hc, cfg->cp_ffn, nqh}) v_ok = v_ok && k % 16 == 0;
            const int pmax = FRAME_MAX_PART / 8;
            v_ok = v_ok && rows(nqkv) * 2 <= pmax && rows(cfg->ffn) * 2 <= pmax && rows(cfg->cp_ffn) * 4 <= pmax &&
                   rows(H) * 2 <= pmax && rows(Hc) * 2 <= pmax && rows(cfg->codec_vocab) <= pmax &&
                   rows(cfg->cp_vocab) <= pmax;
        }
        const bool grid_ok = grid >= cfg->n_kv_heads && v_ok && phases <= FRAME_MAX_PHASES &&
                             cfg->n_kv_heads + 8 <= FRAME_CTL_WORDS && H <= FRAME_MAX_NORM && Hc <= FRAME_MAX_NORM;
        h->frame_ok = h->frame_ok && grid_ok;
        h->frame_grid = grid;
        // talker attention splits: a split's cached K and V fit one ring slot
        const int per_split = (int)(tile / (2 * HD * e));
        h->frame_splits = std::max(1, std::min((cfg->max_ctx + per_split - 1) / per_split,
                                               std::min(16, std::max(1, grid / cfg->n_kv_heads))));
        if (path == Q3_PATH_FRAME && !h->frame_ok) { q3tts_destroy(h); return Q3_ERR_ARG; }
    }
    // split-KV partitions of the talker decode attention: enough blocks to fill
    // the GPU twice at small batch, one split at large batch
    const int blocks = cfg->max_batch * cfg->n_kv_heads;
    int s = std::min((cfg->max_ctx + 31) / 32, (2 * device_sm_count() + blocks - 1) / blocks);
    h->splits_t = std::max(1, std::min(s, MAX_SPLITS));
    // RoPE table: cos, sin of pos * inv_freq_j, inv_freq_j = theta^(-2j/128) in
    // fp32 and the angle formed in fp32 (inv_freq kept fp32 in bf16 models).
    std::vector<float> rope((size_t)L.rope_rows * (HD / 2) * 2);
    for (int p = 0; p < L.rope_rows; ++p)
        for (int j = 0; j < HD / 2; ++j) {
            const float inv = (float)std::pow((double)cfg->rope_theta, -2.0 * j / HD);
            const float ang = (float)p * inv;
            rope[((size_t)p * (HD / 2) + j) * 2 + 0] = (float)std::cos((double)ang);
            rope[((size_t)p * (HD / 2) + j) * 2 + 1] = (float)std::sin((double)ang);
        }
    cudaError_t e = cudaMemcpyAsync(h->p<float>(L.rope), rope.data(), rope.size() * sizeof(float),
                                    cudaMemcpyHostToDevice, h->st);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->p<int>(L.cap_slot), 0xFF, (size_t)cfg->max_batch * sizeof(int), h->st);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->p<int>(L.err), 0, 4 * sizeof(int), h->st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(h->st);
    if (e != cudaSuccess) { q3tts_destroy(h); return Q3_ERR_CUDA; }
    if (upload_frame_params(h) != Q3_OK) { q3tts_destroy(h); return Q3_ERR_CUDA; }
    *out = h;
    return Q3_OK;
}

void q3tts_destroy(q3tts_t* h) {
    if (!h) return;
    if (h->st) cudaStreamSynchronize(h->st);
    invalidate_graph(h);
    if (h->own_stream && h->st) cudaStreamDestroy(h->st);
    delete h;
}

const char* q3tts_last_error(const q3tts_t* h) { return h ? h->last_error.c_str() : "NULL handle"; }

int q3tts_prefill(q3tts_t* h, int batch, const float* prompt, const int32_t* prompt_offsets, const float* text,
                  const int32_t* text_offsets, const float* tts_pad, const q3tts_sampling* rows_in,
                  int32_t* code0_out) {
    if (!h) return Q3_ERR_ARG;
    NvtxRange nvtx("q3tts_prefill");
    const q3tts_config& c = h->c;
    if (batch < 1 || batch > c.max_batch) return fail(h, Q3_ERR_CAPACITY, "batch %d outside 1..%d", batch, c.max_batch);
    if (!prompt || !prompt_offsets || !text_offsets || !tts_pad || !rows_in)
        return fail(h, Q3_ERR_ARG, "NULL argument");
    if (prompt_offsets[0] != 0 || text_offsets[0] != 0) return fail(h, Q3_ERR_ARG, "offsets must start at 0");
    long total_text = 0;
    for (int r = 0; r < batch; ++r) {
        const int len = prompt_offsets[r + 1] - prompt_offsets[r];
        const int nt = text_offsets[r + 1] - text_offsets[r];
        const q3tts_sampling& s = rows_in[r];
        if (len < 1) return fail(h, Q3_ERR_ARG, "row %d: empty prompt", r);
        if (nt < 0) return fail(h, Q3_ERR_ARG, "row %d: negative text count", r);
        if (nt > c.max_text) return fail(h, Q3_ERR_CAPACITY, "row %d: %d text rows > max_text %d", r, nt, c.max_text);
        if (s.max_frames < 0) return fail(h, Q3_ERR_ARG, "row %d: negative max_frames", r);
        if ((long)len + s.max_frames > c.max_ctx)
            return fail(h, Q3_ERR_CAPACITY, "row %d: prompt %d + max_frames %d > max_ctx %d", r, len, s.max_frames,
                        c.max_ctx);
        if ((s.do_sample && !(s.temperature > 0.f)) || (s.cp_do_sample && !(s.cp_temperature > 0.f)))
            return fail(h, Q3_ERR_ARG, "row %d: temperature must be > 0 when sampling", r);
        if (!(s.repetition_penalty > 0.f)) return fail(h, Q3_ERR_ARG, "row %d: repetition_penalty must be > 0", r);
        total_text += nt;
    }
    if (total_text > 0 && !text) return fail(h, Q3_ERR_ARG, "text is NULL but rows have text");

    if (batch != h->graph_batch) invalidate_graph(h);
    h->batch = batch;
    h->prefilled = false;
    h->steps_done = 0;
    const int H = c.hidden;

    // per-row state and settings
    std::vector<RowState> rs(batch);
    std::memset(rs.data(), 0, rs.size() * sizeof(RowState));
    for (int r = 0; r < batch; ++r) {
        rs[r].pos = prompt_offsets[r + 1] - prompt_offsets[r];
        rs[r].code0 = -1;
        rs[r].n_text = text_offsets[r + 1] - text_offsets[r];
        rs[r].text_off = r * c.max_text;
    }
    CK(cudaMemcpyAsync(h->rows(), rs.data(), rs.size() * sizeof(RowState), cudaMemcpyHostToDevice, h->st));
    CK(cudaMemcpyAsync(h->p<q3tts_sampling>(h->L.params), rows_in, (size_t)batch * sizeof(q3tts_sampling),
                       cudaMemcpyHostToDevice, h->st));
    for (int r = 0; r < batch; ++r) {
        const int nt = text_offsets[r + 1] - text_offsets[r];
        if (nt > 0)
            CK(cudaMemcpyAsync(h->p<float>(h->L.text) + (size_t)r * c.max_text * H,
                               text + (size_t)text_offsets[r] * H, (size_t)nt * H * sizeof(float), cudaMemcpyDefault,
                               h->st));
    }
    CK(cudaMemcpyAsync(h->p<float>(h->L.pad), tts_pad, H * sizeof(float), cudaMemcpyDefault, h->st));
    CK(cudaMemsetAsync(h->p<int32_t>(h->L.codes), 0xFF,
                       (size_t)c.max_batch * h->L.frames_cap * MAX_GROUPS * sizeof(int32_t), h->st));
    CK(cudaMemsetAsync(h->err(), 0, 4 * sizeof(int), h->st));
    if (h->frame_ok || h->cl_ok) {
        // exchange words start at epoch 0 (never a live epoch); abort flag and
        // split counters start at 0
        CK(cudaMemsetAsync(h->p<Word>(h->L.fll), 0, h->L.fll_words * sizeof(Word), h->st));
        CK(cudaMemsetAsync(h->p<unsigned>(h->L.fctl), 0, FRAME_CTL_WORDS * sizeof(unsigned), h->st));
    }
    if (h->cl_ok) {
        const ClLayout cl = cl_layout(c);
        CK(cudaMemsetAsync(h->p<Word>(h->L.clxr), 0, cl.xr_words * sizeof(Word), h->st));
        CK(cudaMemsetAsync(h->p<Word>(h->L.cllg), 0, cl.lg_words * sizeof(Word), h->st));
    }

    // prompt through the talker, in chunks of whole tokens across rows
    const int total = prompt_offsets[batch];
    std::vector<int> trow(h->L.mmax), tpos(h->L.mmax), last(h->L.mmax);
    std::vector<int4> tiles;
    tiles.reserve(h->L.mmax);
    std::vector<int> tok_row(total), tok_pos(total);
    for (int r = 0; r < batch; ++r)
        for (int p = prompt_offsets[r]; p < prompt_offsets[r + 1]; ++p) { tok_row[p] = r; tok_pos[p] = p - prompt_offsets[r]; }
    float* x = h->p<float>(h->L.x);
    float* headop = h->p<float>(h->L.headop);
    const int chunk = std::min(PREFILL_CHUNK, h->L.mmax);
    for (int t0 = 0; t0 < total; t0 += chunk) {
        const int M = std::min(chunk, total - t0);
        for (int m = 0; m < M; ++m) {
            const int t = t0 + m;
            trow[m] = tok_row[t];
            tpos[m] = tok_pos[t];
            last[m] = (t + 1 == prompt_offsets[tok_row[t] + 1]) ? tok_row[t] : -1;
        }
        CK(cudaMemcpyAsync(h->p<int>(h->L.t_row), trow.data(), M * sizeof(int), cudaMemcpyHostToDevice, h->st));
        CK(cudaMemcpyAsync(h->p<int>(h->L.t_pos), tpos.data(), M * sizeof(int), cudaMemcpyHostToDevice, h->st));
        CK(cudaMemcpyAsync(h->p<int>(h->L.last_row), last.data(), M * sizeof(int), cudaMemcpyHostToDevice, h->st));
        // attention tiles: runs of up to 64 consecutive tokens of one row
        tiles.clear();
        for (int m = 0; m < M; ++m) {
            if (tiles.empty() || tiles.back().z != trow[m] || tiles.back().y == 64)
                tiles.push_back(make_int4(m, 0, trow[m], tpos[m]));
            tiles.back().y += 1;
        }
        CK(cudaMemcpyAsync(h->p<int4>(h->L.ptiles), tiles.data(), tiles.size() * sizeof(int4), cudaMemcpyHostToDevice,
                           h->st));
        CK(cudaMemcpyAsync(x, prompt + (size_t)t0 * H, (size_t)M * H * sizeof(float), cudaMemcpyDefault, h->st));
        int r = enqueue_layers(h, true, M, x, h->p<int>(h->L.t_row), h->p<int>(h->L.t_pos), h->p<int4>(h->L.ptiles),
                               (int)tiles.size());
        if (r) return r;
        CK(launch_rmsnorm(x, H, M, (const float*)h->w.talker.final_norm, H, c.rms_eps, headop, H,
                          h->p<float>(h->L.h), H, h->p<int>(h->L.last_row), h->st)); debug_wait(h, "launch_rmsnorm");
        // the host vectors are reused by the next chunk: let this chunk's copies finish
        CK(cudaStreamSynchronize(h->st));
    }
    float* logits = h->p<float>(h->L.logits);
    CK(launch_linear(c.dtype, h->w.codec_head, c.codec_vocab, H, headop, H, batch, logits, c.codec_vocab, nullptr, 0,
                     h->tc(), h->err(), h->st)); debug_wait(h, "launch_linear");
    CK(launch_talker_sample(logits, c.codec_vocab, batch, h->rows(), h->p<q3tts_sampling>(h->L.params), c.eos_id,
                            c.suppress_lo, c.suppress_hi, 0, h->err(), h->cap_t, h->p<int>(h->L.cap_slot), h->cap_T,
                            h->st)); debug_wait(h, "launch_talker_sample");
    int err_host[4];
    CK(cudaMemcpyAsync(err_host, h->err(), sizeof err_host, cudaMemcpyDeviceToHost, h->st));
    CK(cudaMemcpyAsync(rs.data(), h->rows(), rs.size() * sizeof(RowState), cudaMemcpyDeviceToHost, h->st));
    CK(cudaStreamSynchronize(h->st));
    if (code0_out) {
        std::vector<int32_t> c0(batch);
        for (int r = 0; r < batch; ++r) c0[r] = rs[r].code0;
        CK(cudaMemcpy(code0_out, c0.data(), batch * sizeof(int32_t), cudaMemcpyDefault));
    }
    h->prefilled = true;
    return read_errors(h, err_host);
}

int q3tts_step_frames(q3tts_t* h, int n_frames, int32_t* codes_out, int32_t* frames_emitted,
                      int32_t* finish_reason) {
    if (!h) return Q3_ERR_ARG;
    NvtxRange nvtx("q3tts_step_frames");
    if (!h->prefilled) return fail(h, Q3_ERR_STATE, "q3tts_step_frames before q3tts_prefill");
    if (n_frames < 0) return fail(h, Q3_ERR_ARG, "negative n_frames");
    const q3tts_config& c = h->c;
    const int B = h->batch;
    if (n_frames > 0 && !h->exec) {
        int r = record_step_graph(h);
        if (r) return r;
    }
    for (int i = 0; i < n_frames; ++i) CK(cudaGraphLaunch(h->exec, h->st));
    const long f0 = h->steps_done;
    if (codes_out && n_frames > 0) {
        cudaPointerAttributes pa;
        const bool dev = cudaPointerGetAttributes(&pa, codes_out) == cudaSuccess &&
                         (pa.type == cudaMemoryTypeDevice || pa.type == cudaMemoryTypeManaged);
        cudaGetLastError();
        const int G = c.n_groups;
        if (dev) {
            CK(launch_pack_codes(h->p<int32_t>(h->L.codes), h->L.frames_cap, f0, n_frames, G, B, codes_out,
                                 (long)n_frames * G, h->st)); debug_wait(h, "launch_pack_codes");
        } else {
            // through the staging area, at most frames_cap frames at a time
            for (long j0 = 0; j0 < n_frames; j0 += h->L.frames_cap) {
                const long nc = std::min((long)h->L.frames_cap, n_frames - j0);
                int32_t* stage = h->p<int32_t>(h->L.codes_stage);
                CK(launch_pack_codes(h->p<int32_t>(h->L.codes), h->L.frames_cap, f0 + j0, (int)nc, G, B, stage,
                                     nc * G, h->st)); debug_wait(h, "launch_pack_codes");
                CK(cudaMemcpy2DAsync(codes_out + j0 * G, (size_t)n_frames * G * sizeof(int32_t), stage,
                                     (size_t)nc * G * sizeof(int32_t), (size_t)nc * G * sizeof(int32_t), B,
                                     cudaMemcpyDeviceToHost, h->st));
            }
        }
    }
    std::vector<RowState> rs(B);
    int err_host[4];
    CK(cudaMemcpyAsync(rs.data(), h->rows(), (size_t)B * sizeof(RowState), cudaMemcpyDeviceToHost, h->st));
    CK(cudaMemcpyAsync(err_host, h->err(), sizeof err_host, cudaMemcpyDeviceToHost, h->st));
    CK(cudaStreamSynchronize(h->st));
    h->steps_done += n_frames;
    for (int r = 0; r < B; ++r) {
        if (frames_emitted) frames_emitted[r] = rs[r].frames;
        if (finish_reason) finish_reason[r] = rs[r].finished ? rs[r].reason : Q3_RUNNING;
    }
    return read_errors(h, err_host);
}

int q3tts_text_embed(q3tts_t* h, int n, const int32_t* ids, float* rows_out) {
    if (!h) return Q3_ERR_ARG;
    NvtxRange nvtx("q3tts_text_embed");
    const q3tts_config& c = h->c;
    if (c.text_vocab <= 0) return fail(h, Q3_ERR_ARG, "the configuration has no text path (text_vocab 0)");
    if (n < 0) return fail(h, Q3_ERR_ARG, "negative n");
    if (n == 0) return Q3_OK;
    if (!ids || !rows_out) return fail(h, Q3_ERR_ARG, "NULL argument");
    auto on_device = [](const void* p) {
        cudaPointerAttributes pa;
        const bool d = cudaPointerGetAttributes(&pa, p) == cudaSuccess &&
                       (pa.type == cudaMemoryTypeDevice || pa.type == cudaMemoryTypeManaged);
        cudaGetLastError();
        return d;
    };
    const bool ids_dev = on_device(ids), out_dev = on_device(rows_out);
    if (!ids_dev)
        for (int i = 0; i < n; ++i)
            if (ids[i] < 0 || ids[i] >= c.text_vocab) return fail(h, Q3_ERR_ARG, "id %d at %d outside [0, %d)", ids[i], i, c.text_vocab);
    const int T = c.text_hidden, H = c.hidden;
    int* dids = h->p<int>(h->L.t_row);          // [mmax] ids of one chunk
    float* e = h->p<float>(h->L.opA);          // [mmax][T] gathered embeddings
    float* a = h->p<float>(h->L.opB);          // [mmax][T] SiLU(fc1)
    float* y = h->p<float>(h->L.x);            // [mmax][H] staging of host-bound rows
    int* err = h->err() + 3;                    // own error word
    CK(cudaMemsetAsync(err, 0, sizeof(int), h->st));
    for (int i0 = 0; i0 < n; i0 += h->L.mmax) {
        const int m = std::min(h->L.mmax, n - i0);
        CK(cudaMemcpyAsync(dids, ids + i0, (size_t)m * sizeof(int), cudaMemcpyDefault, h->st));
        CK(launch_text_gather(c.dtype, h->w.text_emb, dids, m, c.text_vocab, T, e, err, h->st)); debug_wait(h, "launch_text_gather");
        CK(launch_linear(c.dtype, h->w.text_fc1_w, T, T, e, T, m, a, T, (const float*)h->w.text_fc1_b, 0, h->tc(),
                         h->err(), h->st)); debug_wait(h, "launch_linear");
        CK(launch_silu(a, (long)m * T, h->st)); debug_wait(h, "launch_silu");
        float* dst = out_dev ? rows_out + (size_t)i0 * H : y;
        CK(launch_linear(c.dtype, h->w.text_fc2_w, H, T, a, T, m, dst, H, (const float*)h->w.text_fc2_b, 0, h->tc(),
                         h->err(), h->st)); debug_wait(h, "launch_linear");
        if (!out_dev)
            CK(cudaMemcpyAsync(rows_out + (size_t)i0 * H, y, (size_t)m * H * sizeof(float), cudaMemcpyDeviceToHost,
                               h->st));
        // the chunk's buffers are reused by the next one (host ids / rows are read or written in the call)
        CK(cudaStreamSynchronize(h->st));
    }
    int err_host[4] = {0, 0, 0, 0};
    CK(cudaMemcpyAsync(err_host, err, sizeof(int), cudaMemcpyDeviceToHost, h->st));
    CK(cudaStreamSynchronize(h->st));
    return read_errors(h, err_host);
}

int q3tts_set_capture(q3tts_t* h, int n_rows, const int32_t* rows, float* talker_logits, float* cp_logits,
                      int max_frames) {
    if (!h) return Q3_ERR_ARG;
    if (n_rows < 0 || n_rows > h->c.max_batch || (n_rows > 0 && (!rows || !talker_logits || !cp_logits)) ||
        max_frames < 0)
        return fail(h, Q3_ERR_ARG, "bad capture arguments");
    std::vector<int> slot(h->c.max_batch, -1);
    for (int i = 0; i < n_rows; ++i) {
        if (rows[i] < 0 || rows[i] >= h->c.max_batch) return fail(h, Q3_ERR_ARG, "capture row out of range");
        slot[rows[i]] = i;
    }
    CK(cudaMemcpyAsync(h->p<int>(h->L.cap_slot), slot.data(), slot.size() * sizeof(int), cudaMemcpyHostToDevice,
                       h->st));
    CK(cudaStreamSynchronize(h->st));
    h->cap_t = n_rows ? talker_logits : nullptr;
    h->cap_c = n_rows ? cp_logits : nullptr;
    h->cap_T = max_frames;
    invalidate_graph(h);
    return upload_frame_params(h);
}

int q3tts_sample_logits(q3tts_t* h, int n, const float* logits, int talker, const q3tts_sampling* params,
                        const uint8_t* seen, const int32_t* sel_index, int step, const int32_t* noise_row,
                        int32_t* ids_out) {
    if (!h) return Q3_ERR_ARG;
    const q3tts_config& c = h->c;
    if (n < 0 || n > h->L.n_sets) return fail(h, Q3_ERR_ARG, "n must be in 0..%d", h->L.n_sets);
    if (n == 0) return Q3_OK;
    if (!logits || !params || !sel_index || !noise_row || !ids_out) return fail(h, Q3_ERR_ARG, "NULL argument");
    for (int i = 0; i < n; ++i)
        if (!sampling_ok(params[i], talker != 0))
            return fail(h, Q3_ERR_ARG, "set %d: temperature must be > 0 when sampling, repetition_penalty > 0", i);
    const int V = talker ? c.codec_vocab : c.cp_vocab;
    float* lg = h->p<float>(h->L.s_logits);
    uint8_t* sn = seen ? h->p<uint8_t>(h->L.s_seen) : nullptr;
    q3tts_sampling* sp = h->p<q3tts_sampling>(h->L.s_params);
    CK(cudaMemcpyAsync(lg, logits, (size_t)n * V * sizeof(float), cudaMemcpyDefault, h->st));
    if (seen) CK(cudaMemcpyAsync(sn, seen, (size_t)n * V, cudaMemcpyDefault, h->st));
    CK(cudaMemcpyAsync(sp, params, (size_t)n * sizeof(q3tts_sampling), cudaMemcpyHostToDevice, h->st));
    CK(cudaMemcpyAsync(h->p<int>(h->L.s_sel), sel_index, (size_t)n * sizeof(int), cudaMemcpyHostToDevice, h->st));
    CK(cudaMemcpyAsync(h->p<int>(h->L.s_row), noise_row, (size_t)n * sizeof(int), cudaMemcpyHostToDevice, h->st));
    int* serr = h->err() + 2;   // own error word: the frame loop's word is left untouched
    CK(cudaMemsetAsync(serr, 0, sizeof(int), h->st));
    CK(launch_sample_sets(lg, n, V, talker, sp, sn, h->p<int>(h->L.s_sel), step,
                          h->p<int>(h->L.s_row), c.eos_id, c.suppress_lo, c.suppress_hi, h->p<int>(h->L.s_ids),
                          serr, h->st)); debug_wait(h, "launch_sample_sets");
    int err_host[4] = {0, 0, 0, 0};
    CK(cudaMemcpyAsync(ids_out, h->p<int>(h->L.s_ids), (size_t)n * sizeof(int), cudaMemcpyDefault, h->st));
    CK(cudaMemcpyAsync(err_host, serr, sizeof(int), cudaMemcpyDeviceToHost, h->st));
    CK(cudaStreamSynchronize(h->st));
    return read_errors(h, err_host);
}

int q3tts_step_path(const q3tts_t* h, int batch, int* path) {
    if (!h || !path || batch < 1 || batch > h->c.max_batch) return Q3_ERR_ARG;
    *path = batch == 1 && h->cl_ok ? Q3_PATH_CLUSTER : batch == 1 && h->frame_ok ? Q3_PATH_FRAME : Q3_PATH_GRAPH;
    return Q3_OK;
}

int q3tts_step_kernel_count(q3tts_t* h, int* count) {
    if (!h || !count) return Q3_ERR_ARG;
    if (!h->prefilled) return fail(h, Q3_ERR_STATE, "no prefill");
    if (!h->exec) {
        int r = record_step_graph(h);
        if (r) return r;
    }
    size_t n = 0;
    CK(cudaGraphGetNodes(h->graph, nullptr, &n));
    std::vector<cudaGraphNode_t> nodes(n);
    CK(cudaGraphGetNodes(h->graph, nodes.data(), &n));
    int k = 0;
    for (size_t i = 0; i < n; ++i) {
        cudaGraphNodeType t;
        CK(cudaGraphNodeGetType(nodes[i], &t));
        if (t == cudaGraphNodeTypeKernel) ++k;
    }
    *count = k;
    return Q3_OK;
}

}  // extern "C"
