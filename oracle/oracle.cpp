// Oracle for the Qwen3-TTS 12 Hz frame loop -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow CPU restatement of what one frame of the loop computes:
// one talker step (28-layer Qwen3 decoder + codec head + logits processors)
// and the 5-layer code predictor (2-token prefill + 14 autoregressive steps
// with 15 embedding tables and 15 heads).  It exists to check the CUDA path;
// only tests/, the smoke check and the benchmark's CPU-baseline leg may load
// it.  It shares no code, header or table with the CUDA library.
//
// Sources followed (page title, section):
//  * "Qwen3-TTS 移植 ncnn 简明教程" (ncnn discussion 6798), section 1
//    "先搞清楚结构": talker shape (28 layers, GQA 16/8, head_dim 128,
//    QK-Norm, SwiGLU, RMSNorm, codec vocab 3072, eos 2150), predictor
//    (5 layers, 15 tables + 15 heads, table[s-1] / head[s] offset), the input
//    of the next talker step (sum of 16 code embeddings + trailing text, then
//    tts_pad), EOS only on codebook 0, and the three facts (mrope is plain
//    RoPE, config ids, min_new_tokens masks EOS to -inf).
//  * same page, section 6: processor order (repetition penalty ->
//    min-new-tokens -> suppress [2048,3072) except 2150 -> argmax).
//  * "Qwen3-TTS 0.6B CustomVoice 的 pnnx/ncnn 移植..." (ncnn discussion
//    6832), section 3.1: N frames need N+1 talker selections; 3.2: sign-aware
//    repetition penalty, suppression, min_new_tokens, lowest-index argmax
//    ties, NaN fails closed, EOS and max-frame ends recorded apart.
//  * Mizuoto "Qwen3-TTS" engine page, sections "与上游一致的做法" and "速度":
//    processor chain then a multinomial draw done as argmax(p / Exp(1));
//    penalty over a mask of drawn ids; finished rows are fed EOS; q and k are
//    normalised separately; RoPE inv_freq stays fp32 in bf16 models.
//
// Numerics: activations, norms, attention and sums are fp64; weights are the
// fp32 (or bf16-exact) values handed in.  A bf16 model is bf16 in its weights
// and in its K/V cache: every cache entry is rounded to bf16 when stored;
// activations (including every projection's input) stay at full precision.
// Logits are rounded to fp32 before the logits processors, which then run in
// fp32 exactly as specified below.
//
// Parity of end-to-end logits for random-init weights is unpinned beyond the
// invariants the tests check (the pages print no logits for any weights).
#ifdef _OPENMP
#include <omp.h>
#endif
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include <algorithm>

namespace {

enum { DT_F32 = 0, DT_BF16 = 1 };
enum { ERR_OK = 0, ERR_ARG = 1, ERR_NAN = 5 };
enum { REASON_RUNNING = 0, REASON_EOS = 1, REASON_LENGTH = 2 };

}  // namespace

extern "C" {

typedef struct {
    int n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, codec_vocab;
    int cp_layers, cp_hidden, cp_ffn, cp_vocab, n_groups;
    int eos_id, suppress_lo, suppress_hi;
    float rms_eps, rope_theta;
    int dtype;
} oracle_config;

typedef struct {
    const float* attn_norm;   // [L][H]
    const void* wqkv;         // [L][(nq+2nkv)*hd][H]
    const float* q_norm;      // [L][hd]
    const float* k_norm;      // [L][hd]
    const void* wo;           // [L][H][nq*hd]
    const float* mlp_norm;    // [L][H]
    const void* wgu;          // [L][2F][H]
    const void* wd;           // [L][H][F]
    const float* final_norm;  // [H]
} oracle_block;

typedef struct {
    oracle_block talker;
    const void* codec_emb;    // [V][H]
    const void* codec_head;   // [V][H]
    oracle_block cp;
    const void* cp_emb;       // [G-1][cpV][H]
    const void* cp_heads;     // [G-1][cpV][cpH]
    const void* cp_proj_w;    // [cpH][H] or NULL
    const float* cp_proj_b;   // [cpH] or NULL
} oracle_weights;

typedef struct {
    int do_sample;
    float temperature;
    int top_k;
    float top_p;
    float repetition_penalty;
    int min_new_tokens;
    uint64_t seed;
    int max_frames;
    int force_eos_at_frame;
    int cp_do_sample;
    float cp_temperature;
    int cp_top_k;
    float cp_top_p;
} oracle_sampling;

}  // extern "C"

namespace {

// ---------------------------------------------------------------- numbers
double bf16_round(double v) {
    // Round to the nearest bf16 value (8 significant bits), ties to even.
    if (v == 0.0 || !std::isfinite(v)) return v;
    int e;
    std::frexp(v, &e);                       // |v| = m * 2^e, m in [0.5, 1)
    double scale = std::ldexp(1.0, 8 - e);   // puts 8 significant bits left of the point
    double r = std::nearbyint(v * scale) / scale;
    return r;
}

float bf16_bits_to_float(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

struct Mat {  // read-only view of a weight matrix in the model dtype
    const void* p = nullptr;
    int dtype = DT_F32;
    double at(size_t i) const {
        return dtype == DT_F32 ? (double)((const float*)p)[i] : (double)bf16_bits_to_float(((const uint16_t*)p)[i]);
    }
};

// ---------------------------------------------------------------- blocks
// y[n] = x * rsqrt(mean(x^2) + eps) * w[n]
void rmsnorm(const double* x, const float* w, int n, double eps, double* y) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double r = 1.0 / std::sqrt(ss / n + eps);
    for (int i = 0; i < n; ++i) y[i] = x[i] * r * (double)w[i];
}

// Y[m][n] = sum_k W[n][k] * X[m][k]   (W row-major [N][K]); every output
// accumulates over k in increasing order.  With several tokens the running
// sums of all tokens advance together (same order per output, same result).
void linear(const Mat& W, size_t w_off, int N, int K, const double* X, int M, double* Y) {
    if (M == 1) {
        #pragma omp parallel for schedule(static)
        for (int n = 0; n < N; ++n) {
            const size_t row = w_off + (size_t)n * K;
            double acc = 0.0;
            for (int k = 0; k < K; ++k) acc += W.at(row + k) * X[k];
            Y[n] = acc;
        }
        return;
    }
    std::vector<double> Xt((size_t)K * M);   // X transposed: [K][M]
    for (int m = 0; m < M; ++m)
        for (int k = 0; k < K; ++k) Xt[(size_t)k * M + m] = X[(size_t)m * K + k];
    #pragma omp parallel
    {
        std::vector<double> acc(M);
        #pragma omp for schedule(static)
        for (int n = 0; n < N; ++n) {
            const size_t row = w_off + (size_t)n * K;
            std::fill(acc.begin(), acc.end(), 0.0);
            for (int k = 0; k < K; ++k) {
                const double w = W.at(row + k);
                const double* xk = &Xt[(size_t)k * M];
                for (int m = 0; m < M; ++m) acc[m] += w * xk[m];
            }
            for (int m = 0; m < M; ++m) Y[(size_t)m * N + n] = acc[m];
        }
    }
}

double silu(double g) { return g / (1.0 + std::exp(-g)); }

// Rotary embedding, rotate-half convention, at integer position pos.
// inv_freq_j = theta^(-2j/d) held in fp32; angle = pos * inv_freq_j in fp32.
void rope_apply(double* x, int hd, int pos, float theta) {
    const int half = hd / 2;
    for (int j = 0; j < half; ++j) {
        float inv = (float)std::pow((double)theta, -2.0 * j / hd);
        float ang = (float)pos * inv;
        double c = std::cos((double)ang), s = std::sin((double)ang);
        double a = x[j], b = x[j + half];
        x[j] = a * c - b * s;
        x[j + half] = b * c + a * s;
    }
}

// Multimodal RoPE: frequency j rotates by the position of the stream that
// owns it.  mode 0: contiguous sections (sec[0] freqs -> stream 0, next
// sec[1] -> stream 1, rest -> stream 2); mode 1: interleaved (j mod 3).
void mrope_apply(double* x, int hd, const int* pos3, const int* sec, int mode, float theta) {
    const int half = hd / 2;
    for (int j = 0; j < half; ++j) {
        int stream;
        if (mode == 0) stream = j < sec[0] ? 0 : (j < sec[0] + sec[1] ? 1 : 2);
        else stream = j % 3;
        float inv = (float)std::pow((double)theta, -2.0 * j / hd);
        float ang = (float)pos3[stream] * inv;
        double c = std::cos((double)ang), s = std::sin((double)ang);
        double a = x[j], b = x[j + half];
        x[j] = a * c - b * s;
        x[j + half] = b * c + a * s;
    }
}

// Grouped-query attention for one query token over n cached positions.
// q [nq][hd]; K, V [nkv][cap][hd] (first n used); q head h reads kv head h/(nq/nkv).
void gqa_attend(const double* q, const double* K, const double* V, int cap, int n, int nq, int nkv, int hd,
                double* out) {
    const int group = nq / nkv;
    const double scale = 1.0 / std::sqrt((double)hd);
    std::vector<double> s(n);
    for (int h = 0; h < nq; ++h) {
        const int g = h / group;
        const double* Kg = K + (size_t)g * cap * hd;
        const double* Vg = V + (size_t)g * cap * hd;
        double mx = -INFINITY;
        for (int j = 0; j < n; ++j) {
            double d = 0.0;
            for (int i = 0; i < hd; ++i) d += q[h * hd + i] * Kg[(size_t)j * hd + i];
            s[j] = d * scale;
            mx = std::max(mx, s[j]);
        }
        double z = 0.0;
        for (int j = 0; j < n; ++j) { s[j] = std::exp(s[j] - mx); z += s[j]; }
        for (int i = 0; i < hd; ++i) {
            double acc = 0.0;
            for (int j = 0; j < n; ++j) acc += s[j] * Vg[(size_t)j * hd + i];
            out[h * hd + i] = acc / z;
        }
    }
}

// ---------------------------------------------------------------- sampler
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): 10 rounds of the
// multiply-xor bijection with a Weyl-incremented key.
void philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; ++r) {
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

// ln 2 split for the exponential's argument reduction: LN2_HI keeps the top
// 16 significant bits so that n * LN2_HI is exact for |n| < 2^8.
const float LN2_HI = 0.693145751953125f;          // 0x3F317200
const float LN2_LO = 1.428606765330187e-06f;      // ln2 - LN2_HI rounded to fp32
const float INV_LN2 = 1.44269502162933349609375f;  // 1/ln2 rounded to fp32

// exp(x) for x <= 0, fp32, IEEE + - * only (no FMA): Cody-Waite reduction
// x = n ln2 + r, Taylor series of e^r to degree 8 in Horner form, times 2^n.
float spec_expf(float x) {
    if (x < -86.0f) return 0.0f;
    float n = std::nearbyint(x * INV_LN2);
    float r = (x - n * LN2_HI) - n * LN2_LO;
    float p = 1.0f / 40320.0f;
    p = 1.0f / 5040.0f + r * p;
    p = 1.0f / 720.0f + r * p;
    p = 1.0f / 120.0f + r * p;
    p = 1.0f / 24.0f + r * p;
    p = 1.0f / 6.0f + r * p;
    p = 0.5f + r * p;
    p = 1.0f + r * p;
    p = 1.0f + r * p;
    int ni = (int)n;
    uint32_t bits = (uint32_t)(ni + 127) << 23;
    float two_n;
    std::memcpy(&two_n, &bits, 4);
    return p * two_n;
}

// log(u) for u in (0, 1), fp32, IEEE + - * / only (no FMA):
// u = f * 2^e with f in [sqrt(1/2), sqrt(2)); log f = 2 atanh(t), t = (f-1)/(f+1),
// atanh series to t^9; log u = e*LN2_LO + log f + e*LN2_HI.
float spec_logf(float u) {
    uint32_t bits;
    std::memcpy(&bits, &u, 4);
    int e = (int)((bits >> 23) & 0xFF) - 126;       // u = f * 2^e, f in [0.5, 1)
    uint32_t fb = (bits & 0x007FFFFFu) | 0x3F000000u;
    float f;
    std::memcpy(&f, &fb, 4);
    if (f < 0.70710678f) { f = f * 2.0f; e = e - 1; }
    float t = (f - 1.0f) / (f + 1.0f);
    float s = t * t;
    float p = 2.0f / 9.0f;
    p = 2.0f / 7.0f + s * p;
    p = 2.0f / 5.0f + s * p;
    p = 2.0f / 3.0f + s * p;
    p = 2.0f + s * p;
    float lf = t * p;
    float ef = (float)e;
    return (ef * LN2_LO + lf) + ef * LN2_HI;
}

// Uniform in (0,1) for (row, frame, step, token) under a row seed:
// counter = (token, step, frame, row), key = (seed lo, seed hi);
// u = (2 * (x0 >> 9) + 1) * 2^-24 (exact in fp32).
float noise_uniform(uint64_t seed, uint32_t row, uint32_t frame, uint32_t step, uint32_t token) {
    uint32_t ctr[4] = {token, step, frame, row};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t o[4];
    philox4x32_10(ctr, key, o);
    uint32_t m = o[0] >> 9;
    return (float)(2u * m + 1u) * (1.0f / 16777216.0f);
}

struct SampleParams {
    int do_sample;
    float temperature;
    int top_k;
    float top_p;
};

// Logits processors and the draw for one selection.
//   talker: repetition penalty over `seen`, EOS -> -inf while sel < min_new,
//   suppress [sup_lo, sup_hi) except eos.  Then greedy argmax, or
//   temperature -> top-k -> top-p -> argmax over kept ids of w_i / E_i with
//   w_i = exp(l_i - max) and E_i = -log(u_i) (one Exp(1) draw per id).
// Returns ERR_NAN if any input logit is NaN or +inf, or no logit is finite
// (no id is chosen then).
int sample_one(const float* logits_in, int V, const SampleParams& sp, bool talker, float penalty,
               const uint8_t* seen, int sel_index, int min_new, int eos, int sup_lo, int sup_hi,
               uint64_t seed, uint32_t row, uint32_t frame, uint32_t step, int* out_id, double* out_margin,
               float* processed_out) {
    std::vector<float> l(logits_in, logits_in + V);
    for (int i = 0; i < V; ++i)
        if (std::isnan(l[i]) || l[i] == INFINITY) return ERR_NAN;
    if (talker) {
        if (penalty != 1.0f && seen)
            for (int i = 0; i < V; ++i)
                if (seen[i]) l[i] = l[i] < 0.0f ? l[i] * penalty : l[i] / penalty;
        if (sel_index < min_new && eos >= 0 && eos < V) l[eos] = -INFINITY;
        for (int i = std::max(sup_lo, 0); i < std::min(sup_hi, V); ++i)
            if (i != eos) l[i] = -INFINITY;
    }
    if (processed_out) std::memcpy(processed_out, l.data(), sizeof(float) * V);

    if (!sp.do_sample) {
        int best = 0;
        for (int i = 1; i < V; ++i)
            if (l[i] > l[best]) best = i;
        double second = -INFINITY;
        for (int i = 0; i < V; ++i)
            if (i != best && l[i] > second) second = l[i];
        *out_id = best;
        *out_margin = (double)l[best] - second;
        return ERR_OK;
    }

    if (sp.temperature != 1.0f)
        for (int i = 0; i < V; ++i) l[i] = l[i] / sp.temperature;

    // top-k: keep every logit >= the k-th largest (ties kept)
    float vk = -INFINITY;
    if (sp.top_k > 0 && sp.top_k < V) {
        std::vector<float> sorted(l);
        std::sort(sorted.begin(), sorted.end(), [](float a, float b) { return a > b; });
        vk = sorted[sp.top_k - 1];
    }
    std::vector<int> kept;
    for (int i = 0; i < V; ++i)
        if (l[i] != -INFINITY && l[i] >= vk) kept.push_back(i);
    if (kept.empty()) return ERR_NAN;
    std::sort(kept.begin(), kept.end(), [&](int a, int b) { return l[a] > l[b] || (l[a] == l[b] && a < b); });
    const float mx = l[kept[0]];
    std::vector<float> w(V, 0.0f);
    for (int i = 0; i < V; ++i)
        if (l[i] != -INFINITY) w[i] = spec_expf(l[i] - mx);

    // top-p: fixed-point weights W_i = floor(w_i * 2^40), exact sums in the
    // (l desc, id asc) order; keep j iff j == 0 or C_j < top_p * Z
    std::vector<double> cum_ratio(V, 0.0);   // C_j / (top_p Z) of each kept id, for the margin
    if (sp.top_p < 1.0f) {
        std::vector<int64_t> W(V, 0);
        int64_t Z = 0;
        for (int i : kept) { W[i] = (int64_t)std::floor((double)w[i] * 1099511627776.0); Z += W[i]; }
        const double limit = (double)sp.top_p * (double)Z;
        std::vector<int> nk;
        int64_t C = 0;
        for (size_t j = 0; j < kept.size(); ++j) {
            cum_ratio[kept[j]] = limit > 0 ? (double)C / limit : 0.0;
            if (j == 0 || (double)C < limit) nk.push_back(kept[j]);
            C += W[kept[j]];
        }
        kept.swap(nk);
    }

    // draw: argmax of w_i / E_i over the kept ids, lowest id on ties
    auto score = [&](int i) {
        const float u = noise_uniform(seed, row, frame, step, (uint32_t)i);
        return w[i] / -spec_logf(u);
    };
    int best = -1;
    float bs = 0.0f;
    std::vector<int> by_id(kept);
    std::sort(by_id.begin(), by_id.end());
    for (int i : by_id) {
        const float sc = score(i);
        if (best < 0 || sc > bs) { best = i; bs = sc; }
    }
    *out_id = best;

    // Decision margin (in processed-logit units, ~ natural-log units of the
    // score): the winner must beat, by the margin, every id that a small logit
    // perturbation could keep -- the kept ids and the ids within the margin of
    // the top-k or top-p boundary -- and must not itself sit near a boundary.
    const double near = 0.05;
    double margin = INFINITY;
    auto near_top_p = [&](int i) {
        return sp.top_p < 1.0f && cum_ratio[i] > 0.0 && std::fabs(std::log(cum_ratio[i])) < near;
    };
    for (int i = 0; i < V; ++i) {
        if (i == best || l[i] == -INFINITY) continue;
        const bool kept_i = std::binary_search(by_id.begin(), by_id.end(), i);
        const bool cand = kept_i || (vk != -INFINITY && (double)l[i] >= (double)vk - near) || near_top_p(i);
        if (!cand) continue;
        margin = std::min(margin, std::log((double)bs / (double)score(i)));
    }
    if (vk != -INFINITY) {
        // the winner drops out of top-k if the next value below it rises past it
        float below = -INFINITY;
        for (int i = 0; i < V; ++i)
            if (l[i] < vk && l[i] > below) below = l[i];
        if (below != -INFINITY) margin = std::min(margin, (double)l[best] - (double)below);
    }
    if (near_top_p(best)) margin = std::min(margin, std::fabs(std::log(cum_ratio[best])));
    *out_margin = margin;
    return ERR_OK;
}

// ---------------------------------------------------------------- model
struct Block {
    const oracle_block* w;
    int L, H, nq, nkv, hd, F;
    Mat wqkv, wo, wgu, wd;
};

struct Row {
    int prompt_len = 0;
    int pos = 0;               // next talker position
    int sel = 0;               // number of talker selections made
    int code0 = -1;            // last talker selection
    std::vector<double> h;     // post-final-norm talker hidden at the last selection
    std::vector<double> K, V;  // talker cache [L][nkv][cap][hd]
    std::vector<double> cK, cV;// predictor cache [cpL][nkv][16][hd]
    std::vector<uint8_t> seen; // ids drawn so far (codebook 0)
    std::vector<double> text;  // trailing text rows [n_text][H]
    int n_text = 0;
    int frames = 0;
    int finished = 0;
    int reason = REASON_RUNNING;
    oracle_sampling sp{};
    uint32_t row_id = 0;
    long n_selections = 0;
    long n_predictor_runs = 0;
};

struct Oracle {
    oracle_config c;
    oracle_weights w;
    Block talker, cp;
    Mat codec_emb, codec_head, cp_emb, cp_heads, cp_proj_w;
    int batch = 0, cap = 0, T = 0;
    bool capture = false;
    std::vector<Row> rows;
    std::vector<double> pad;
    // per row outputs, absolute frame indexing; selection k in [0, T]
    std::vector<int32_t> own_sel, used_codes, own_cp;
    std::vector<double> sel_margin, cp_margin;
    std::vector<float> talker_logits, cp_logits;

    // projection inputs are not rounded (weights and the K/V cache carry the model dtype)
    double operand(double v) const { return v; }
    double kvstore(double v) const { return c.dtype == DT_BF16 ? bf16_round(v) : (double)(float)v; }
};

void make_block(Block& b, const oracle_block* w, int L, int H, const oracle_config& c, int F) {
    b.w = w; b.L = L; b.H = H; b.nq = c.n_q_heads; b.nkv = c.n_kv_heads; b.hd = c.head_dim; b.F = F;
    b.wqkv = {w->wqkv, c.dtype}; b.wo = {w->wo, c.dtype}; b.wgu = {w->wgu, c.dtype}; b.wd = {w->wd, c.dtype};
}

// One decoder layer over M consecutive tokens of one sequence at positions
// p0 .. p0+M-1 (causal).  x [M][H] is the residual stream (updated in place).
// K, V: this layer's cache [nkv][cap][hd].
void layer_forward(const Oracle& o, const Block& b, int l, double* x, int M, int p0, double* K, double* V, int cap) {
    const int H = b.H, hd = b.hd, nq = b.nq, nkv = b.nkv, F = b.F;
    const int nqkv = (nq + 2 * nkv) * hd;
    const double eps = o.c.rms_eps;
    std::vector<double> xn((size_t)M * H), qkv((size_t)M * nqkv), att((size_t)M * nq * hd);
    std::vector<double> y((size_t)M * H), gu((size_t)M * 2 * F), act((size_t)M * F);

    // attention block
    for (int m = 0; m < M; ++m) {
        rmsnorm(x + (size_t)m * H, b.w->attn_norm + (size_t)l * H, H, eps, &xn[(size_t)m * H]);
        for (int i = 0; i < H; ++i) xn[(size_t)m * H + i] = o.operand(xn[(size_t)m * H + i]);
    }
    linear(b.wqkv, (size_t)l * nqkv * H, nqkv, H, xn.data(), M, qkv.data());
    const float* qn = b.w->q_norm + (size_t)l * hd;
    const float* kn = b.w->k_norm + (size_t)l * hd;
    std::vector<double> tmp(hd);
    for (int m = 0; m < M; ++m) {
        double* t = &qkv[(size_t)m * nqkv];
        const int pos = p0 + m;
        for (int h = 0; h < nq; ++h) {           // q heads: QK-norm then RoPE
            rmsnorm(t + h * hd, qn, hd, eps, tmp.data());
            rope_apply(tmp.data(), hd, pos, o.c.rope_theta);
            std::memcpy(t + h * hd, tmp.data(), sizeof(double) * hd);
        }
        for (int g = 0; g < nkv; ++g) {          // k heads: QK-norm, RoPE, cache; v heads: cache
            double* kh = t + (nq + g) * hd;
            double* vh = t + (nq + nkv + g) * hd;
            rmsnorm(kh, kn, hd, eps, tmp.data());
            rope_apply(tmp.data(), hd, pos, o.c.rope_theta);
            for (int i = 0; i < hd; ++i) {
                K[((size_t)g * cap + pos) * hd + i] = o.kvstore(tmp[i]);
                V[((size_t)g * cap + pos) * hd + i] = o.kvstore(vh[i]);
            }
        }
    }
    for (int m = 0; m < M; ++m)
        gqa_attend(&qkv[(size_t)m * nqkv], K, V, cap, p0 + m + 1, nq, nkv, hd, &att[(size_t)m * nq * hd]);
    for (auto& v : att) v = o.operand(v);
    linear(b.wo, (size_t)l * H * nq * hd, H, nq * hd, att.data(), M, y.data());
    for (size_t i = 0; i < (size_t)M * H; ++i) x[i] += y[i];

    // MLP block
    for (int m = 0; m < M; ++m) {
        rmsnorm(x + (size_t)m * H, b.w->mlp_norm + (size_t)l * H, H, eps, &xn[(size_t)m * H]);
        for (int i = 0; i < H; ++i) xn[(size_t)m * H + i] = o.operand(xn[(size_t)m * H + i]);
    }
    linear(b.wgu, (size_t)l * 2 * F * H, 2 * F, H, xn.data(), M, gu.data());
    for (int m = 0; m < M; ++m)
        for (int i = 0; i < F; ++i)
            act[(size_t)m * F + i] = o.operand(silu(gu[(size_t)m * 2 * F + i]) * gu[(size_t)m * 2 * F + F + i]);
    linear(b.wd, (size_t)l * H * F, H, F, act.data(), M, y.data());
    for (size_t i = 0; i < (size_t)M * H; ++i) x[i] += y[i];
}

// Talker over M tokens of row r starting at its current position; returns
// the post-final-norm hidden of the last token in h_out and its fp32 logits.
void talker_forward(Oracle& o, Row& r, double* x, int M, double* h_out, float* logits) {
    const Block& b = o.talker;
    const size_t lstride = (size_t)b.nkv * o.cap * b.hd;
    for (int l = 0; l < b.L; ++l)
        layer_forward(o, b, l, x, M, r.pos, &r.K[l * lstride], &r.V[l * lstride], o.cap);
    r.pos += M;
    rmsnorm(x + (size_t)(M - 1) * b.H, b.w->final_norm, b.H, o.c.rms_eps, h_out);
    std::vector<double> hn(b.H), lg(o.c.codec_vocab);
    for (int i = 0; i < b.H; ++i) hn[i] = o.operand(h_out[i]);
    linear(o.codec_head, 0, o.c.codec_vocab, b.H, hn.data(), 1, lg.data());
    for (int i = 0; i < o.c.codec_vocab; ++i) logits[i] = (float)lg[i];
}

// Predictor input token: a talker-width vector, projected to predictor width
// when the widths differ (weight + bias).
void cp_input(const Oracle& o, const double* v, double* out) {
    const int H = o.c.hidden, Hc = o.c.cp_hidden;
    if (H == Hc) { std::memcpy(out, v, sizeof(double) * H); return; }
    std::vector<double> vin(H);
    for (int i = 0; i < H; ++i) vin[i] = o.operand(v[i]);
    linear(o.cp_proj_w, 0, Hc, H, vin.data(), 1, out);
    for (int i = 0; i < Hc; ++i) out[i] += (double)o.w.cp_proj_b[i];
}

// Predictor layers over M tokens at positions p0..; then final norm of the last
// token and head[s] -> fp32 logits.
void cp_forward(Oracle& o, Row& r, double* x, int M, int p0, int head, float* logits) {
    const Block& b = o.cp;
    const size_t lstride = (size_t)b.nkv * 16 * b.hd;
    for (int l = 0; l < b.L; ++l)
        layer_forward(o, b, l, x, M, p0, &r.cK[l * lstride], &r.cV[l * lstride], 16);
    std::vector<double> hn(b.H), lg(o.c.cp_vocab);
    rmsnorm(x + (size_t)(M - 1) * b.H, b.w->final_norm, b.H, o.c.rms_eps, hn.data());
    for (auto& v : hn) v = o.operand(v);
    linear(o.cp_heads, (size_t)head * o.c.cp_vocab * b.H, o.c.cp_vocab, b.H, hn.data(), 1, lg.data());
    for (int i = 0; i < o.c.cp_vocab; ++i) logits[i] = (float)lg[i];
}

void emb_row(const Mat& t, size_t row, int H, double* out) {
    for (int i = 0; i < H; ++i) out[i] = t.at(row * H + i);
}

int talker_select(Oracle& o, int ri, Row& r, const float* logits, int k, const int32_t* teacher_sel) {
    const int V = o.c.codec_vocab;
    SampleParams sp{r.sp.do_sample, r.sp.temperature, r.sp.top_k, r.sp.top_p};
    int id = 0;
    double margin = 0.0;
    int err = sample_one(logits, V, sp, true, r.sp.repetition_penalty, r.seen.data(), k, r.sp.min_new_tokens,
                         o.c.eos_id, o.c.suppress_lo, o.c.suppress_hi, r.sp.seed, r.row_id, (uint32_t)k, 0, &id,
                         &margin, nullptr);
    if (err) return err;
    const size_t at = (size_t)ri * (o.T + 1) + k;
    o.own_sel[at] = id;
    o.sel_margin[at] = margin;
    if (o.capture) std::memcpy(&o.talker_logits[at * V], logits, sizeof(float) * V);
    if (r.sp.force_eos_at_frame >= 0 && k == r.sp.force_eos_at_frame) id = o.c.eos_id;
    if (teacher_sel) id = *teacher_sel;
    r.code0 = id;
    r.sel = k + 1;
    r.n_selections++;
    if (id >= 0 && id < V) r.seen[id] = 1;
    if (id == o.c.eos_id) { r.finished = 1; r.reason = REASON_EOS; r.frames = k; }
    else if (k >= r.sp.max_frames) { r.finished = 1; r.reason = REASON_LENGTH; r.frames = k; }
    return ERR_OK;
}

}  // namespace

extern "C" {

void* oracle_create(const oracle_config* c, const oracle_weights* w, int batch, int max_ctx, int max_frames,
                    int capture_logits) {
    if (!c || !w || batch <= 0 || max_ctx <= 0 || max_frames < 0) return nullptr;
    if (c->n_q_heads % c->n_kv_heads != 0 || c->head_dim % 2 != 0) return nullptr;
    Oracle* o = new Oracle();
    o->c = *c;
    o->w = *w;
    make_block(o->talker, &o->w.talker, c->n_layers, c->hidden, *c, c->ffn);
    make_block(o->cp, &o->w.cp, c->cp_layers, c->cp_hidden, *c, c->cp_ffn);
    o->codec_emb = {w->codec_emb, c->dtype};
    o->codec_head = {w->codec_head, c->dtype};
    o->cp_emb = {w->cp_emb, c->dtype};
    o->cp_heads = {w->cp_heads, c->dtype};
    o->cp_proj_w = {w->cp_proj_w, c->dtype};
    o->batch = batch;
    o->cap = max_ctx;
    o->T = max_frames;
    o->capture = capture_logits != 0;
    const int G1 = c->n_groups - 1;
    o->own_sel.assign((size_t)batch * (max_frames + 1), -1);
    o->sel_margin.assign((size_t)batch * (max_frames + 1), 0.0);
    o->used_codes.assign((size_t)batch * max_frames * c->n_groups, -1);
    o->own_cp.assign((size_t)batch * max_frames * G1, -1);
    o->cp_margin.assign((size_t)batch * max_frames * G1, 0.0);
    if (o->capture) {
        o->talker_logits.assign((size_t)batch * (max_frames + 1) * c->codec_vocab, 0.0f);
        o->cp_logits.assign((size_t)batch * max_frames * G1 * c->cp_vocab, 0.0f);
    }
    return o;
}

void oracle_destroy(void* h) { delete (Oracle*)h; }

// Text side ("Qwen3-TTS 移植 ncnn 简明教程" section 1, talker bullet: BPE ids
// -> 2048-d text embedding -> ResizeMLP(2048 -> 2048 -> talker width) with
// SiLU between its two linear layers): for each id, in this order,
//   e = emb[id];  a = silu(W1 e + b1);  out = W2 a + b2   (fp64).
// Returns ERR_ARG for an id outside [0, vocab).
int oracle_text_embed(const void* emb, const void* w1, const float* b1, const void* w2, const float* b2, int dtype,
                      int vocab, int T, int H, const int32_t* ids, int n, double* out) {
    const Mat E{emb, dtype}, W1{w1, dtype}, W2{w2, dtype};
    std::vector<double> e(T), a(T);
    for (int i = 0; i < n; ++i) {
        const int id = ids[i];
        if (id < 0 || id >= vocab) return ERR_ARG;
        for (int k = 0; k < T; ++k) e[k] = E.at((size_t)id * T + k);
        for (int j = 0; j < T; ++j) {
            double acc = 0.0;
            for (int k = 0; k < T; ++k) acc += W1.at((size_t)j * T + k) * e[k];
            a[j] = silu(acc + (double)b1[j]);
        }
        for (int j = 0; j < H; ++j) {
            double acc = 0.0;
            for (int k = 0; k < T; ++k) acc += W2.at((size_t)j * T + k) * a[k];
            out[(size_t)i * H + j] = acc + (double)b2[j];
        }
    }
    return ERR_OK;
}

// Worker threads of the parallel loops from now on (timing only; results do
// not depend on it); returns the count in effect before the call.
int oracle_set_threads(int n) {
#ifdef _OPENMP
    const int old = omp_get_max_threads();
    if (n > 0) omp_set_num_threads(n);
    return old;
#else
    (void)n;
    return 1;
#endif
}

// Prefill: prompt rows through the talker, then selection 0 of each row.
// row_ids: the row index each row uses in the noise counter.
int oracle_prefill(void* h, const float* prompt, const int32_t* prompt_off, const float* text,
                   const int32_t* text_off, const float* tts_pad, const oracle_sampling* sp, const int32_t* row_ids,
                   const int32_t* teacher /* [batch][T+1][G] or NULL */) {
    Oracle& o = *(Oracle*)h;
    const int H = o.c.hidden, hd = o.c.head_dim, nkv = o.c.n_kv_heads;
    o.rows.assign(o.batch, Row());
    o.pad.assign(tts_pad, tts_pad + H);
    for (int ri = 0; ri < o.batch; ++ri) {
        Row& r = o.rows[ri];
        r.sp = sp[ri];
        r.row_id = (uint32_t)row_ids[ri];
        r.prompt_len = prompt_off[ri + 1] - prompt_off[ri];
        if (r.prompt_len <= 0 || r.prompt_len + r.sp.max_frames > o.cap || r.sp.max_frames > o.T) return ERR_ARG;
        r.K.assign((size_t)o.c.n_layers * nkv * o.cap * hd, 0.0);
        r.V.assign(r.K.size(), 0.0);
        r.cK.assign((size_t)o.c.cp_layers * nkv * 16 * hd, 0.0);
        r.cV.assign(r.cK.size(), 0.0);
        r.seen.assign(o.c.codec_vocab, 0);
        r.h.assign(H, 0.0);
        r.n_text = text_off[ri + 1] - text_off[ri];
        r.text.assign(text + (size_t)text_off[ri] * H, text + (size_t)text_off[ri + 1] * H);
        std::vector<double> x(prompt + (size_t)prompt_off[ri] * H, prompt + (size_t)prompt_off[ri + 1] * H);
        std::vector<float> logits(o.c.codec_vocab);
        talker_forward(o, r, x.data(), r.prompt_len, r.h.data(), logits.data());
        const int32_t* tsel = teacher ? &teacher[(size_t)ri * (o.T + 1) * o.c.n_groups] : nullptr;
        int err = talker_select(o, ri, r, logits.data(), 0, tsel);
        if (err) return err;
    }
    return ERR_OK;
}

// Run n talker steps on every unfinished row.  Step k completes frame k-1
// (predictor on the pending code0 and the hidden that chose it), assembles the
// next talker input and makes selection k.
int oracle_step(void* h, int n, const int32_t* teacher /* [batch][T+1][G] or NULL */) {
    Oracle& o = *(Oracle*)h;
    const int H = o.c.hidden, Hc = o.c.cp_hidden, G = o.c.n_groups, G1 = G - 1;
    const int cpV = o.c.cp_vocab;
    for (int ri = 0; ri < o.batch; ++ri) {
        Row& r = o.rows[ri];
        for (int it = 0; it < n && !r.finished; ++it) {
            const int k = r.sel;           // this step makes selection k
            const int f = k - 1;           // and completes frame f
            const int32_t* trow = teacher ? &teacher[((size_t)ri * (o.T + 1)) * G] : nullptr;
            int32_t* codes = &o.used_codes[((size_t)ri * o.T + f) * G];
            if (r.code0 < 0 || r.code0 >= o.c.codec_vocab) return ERR_ARG;
            codes[0] = r.code0;

            // code predictor: tokens [h, codec_emb(code0)] at positions 0,1, then
            // table[s-1](code_s) at position s+1 -> head[s] -> code s+1.
            std::vector<double> xin((size_t)2 * Hc), tok(H);
            cp_input(o, r.h.data(), &xin[0]);
            emb_row(o.codec_emb, (size_t)r.code0, H, tok.data());
            cp_input(o, tok.data(), &xin[Hc]);
            std::vector<float> lg(cpV);
            SampleParams cps{r.sp.cp_do_sample, r.sp.cp_temperature, r.sp.cp_top_k, r.sp.cp_top_p};
            for (int s = 0; s < G1; ++s) {
                if (s == 0) {
                    cp_forward(o, r, xin.data(), 2, 0, 0, lg.data());
                } else {
                    if (codes[s] < 0 || codes[s] >= cpV) return ERR_ARG;
                    emb_row(o.cp_emb, (size_t)(s - 1) * cpV + codes[s], H, tok.data());
                    std::vector<double> x1(Hc);
                    cp_input(o, tok.data(), x1.data());
                    cp_forward(o, r, x1.data(), 1, s + 1, s, lg.data());
                }
                int id = 0;
                double margin = 0.0;
                int err = sample_one(lg.data(), cpV, cps, false, 1.0f, nullptr, 0, 0, -1, 0, 0, r.sp.seed,
                                     r.row_id, (uint32_t)f, (uint32_t)(s + 1), &id, &margin, nullptr);
                if (err) return err;
                const size_t at = ((size_t)ri * o.T + f) * G1 + s;
                o.own_cp[at] = id;
                o.cp_margin[at] = margin;
                if (o.capture) std::memcpy(&o.cp_logits[at * cpV], lg.data(), sizeof(float) * cpV);
                codes[s + 1] = trow ? trow[(size_t)f * G + s + 1] : id;
            }
            r.n_predictor_runs++;
            r.frames = k;

            // next talker input: codec_emb(code0) + sum_q table[q-1](code_q) + text
            std::vector<double> x(H);
            emb_row(o.codec_emb, (size_t)codes[0], H, x.data());
            for (int q = 1; q < G; ++q) {
                if (codes[q] < 0 || codes[q] >= cpV) return ERR_ARG;
                emb_row(o.cp_emb, (size_t)(q - 1) * cpV + codes[q], H, tok.data());
                for (int i = 0; i < H; ++i) x[i] += tok[i];
            }
            const double* text_row = (k - 1 < r.n_text) ? &r.text[(size_t)(k - 1) * H] : o.pad.data();
            for (int i = 0; i < H; ++i) x[i] += text_row[i];

            std::vector<float> logits(o.c.codec_vocab);
            talker_forward(o, r, x.data(), 1, r.h.data(), logits.data());
            const int32_t* tsel = trow ? &trow[(size_t)k * G] : nullptr;
            int err = talker_select(o, ri, r, logits.data(), k, tsel);
            if (err) return err;
        }
    }
    return ERR_OK;
}

// Copy out per-row results.  what: 0 own_sel [B][T+1], 1 sel_margin [B][T+1] (f64),
// 2 used codes [B][T][G], 3 own_cp [B][T][G-1], 4 cp_margin [B][T][G-1] (f64),
// 5 talker logits [B][T+1][V] (f32), 6 cp logits [B][T][G-1][cpV] (f32),
// 7 frames [B], 8 finish reason [B], 9 selections [B] (i64), 10 predictor runs [B] (i64).
int oracle_get(void* h, int what, void* out) {
    Oracle& o = *(Oracle*)h;
    auto cp = [&](const void* src, size_t bytes) { std::memcpy(out, src, bytes); return ERR_OK; };
    switch (what) {
        case 0: return cp(o.own_sel.data(), o.own_sel.size() * 4);
        case 1: return cp(o.sel_margin.data(), o.sel_margin.size() * 8);
        case 2: return cp(o.used_codes.data(), o.used_codes.size() * 4);
        case 3: return cp(o.own_cp.data(), o.own_cp.size() * 4);
        case 4: return cp(o.cp_margin.data(), o.cp_margin.size() * 8);
        case 5: return o.capture ? cp(o.talker_logits.data(), o.talker_logits.size() * 4) : ERR_ARG;
        case 6: return o.capture ? cp(o.cp_logits.data(), o.cp_logits.size() * 4) : ERR_ARG;
        default: break;
    }
    for (int ri = 0; ri < o.batch; ++ri) {
        const Row& r = o.rows[ri];
        if (what == 7) ((int32_t*)out)[ri] = r.frames;
        else if (what == 8) ((int32_t*)out)[ri] = r.reason;
        else if (what == 9) ((int64_t*)out)[ri] = r.n_selections;
        else if (what == 10) ((int64_t*)out)[ri] = r.n_predictor_runs;
        else return ERR_ARG;
    }
    return ERR_OK;
}

// ------------------------------------------------------------ unit entry points
int oracle_sample(const float* logits, int V, const oracle_sampling* sp, int talker, const uint8_t* seen,
                  int sel_index, int eos, int sup_lo, int sup_hi, uint32_t row, uint32_t frame, uint32_t step,
                  int* out_id, double* out_margin, float* processed_out) {
    SampleParams p = talker ? SampleParams{sp->do_sample, sp->temperature, sp->top_k, sp->top_p}
                            : SampleParams{sp->cp_do_sample, sp->cp_temperature, sp->cp_top_k, sp->cp_top_p};
    return sample_one(logits, V, p, talker != 0, sp->repetition_penalty, seen, sel_index, sp->min_new_tokens, eos,
                      sup_lo, sup_hi, sp->seed, row, frame, step, out_id, out_margin, processed_out);
}

void oracle_philox(const uint32_t* ctr, const uint32_t* key, uint32_t* out) { philox4x32_10(ctr, key, out); }
float oracle_spec_expf(float x) { return spec_expf(x); }
float oracle_spec_logf(float u) { return spec_logf(u); }
float oracle_noise_uniform(uint64_t seed, uint32_t row, uint32_t frame, uint32_t step, uint32_t token) {
    return noise_uniform(seed, row, frame, step, token);
}
double oracle_bf16_round(double v) { return bf16_round(v); }
void oracle_rmsnorm(const double* x, const float* w, int n, double eps, double* y) { rmsnorm(x, w, n, eps, y); }
void oracle_rope(double* x, int hd, int pos, float theta) { rope_apply(x, hd, pos, theta); }
void oracle_mrope(double* x, int hd, const int* pos3, const int* sec, int mode, float theta) {
    mrope_apply(x, hd, pos3, sec, mode, theta);
}
void oracle_attend(const double* q, const double* K, const double* V, int cap, int n, int nq, int nkv, int hd,
                   double* out) {
    gqa_attend(q, K, V, cap, n, nq, nkv, hd, out);
}

}  // extern "C"
