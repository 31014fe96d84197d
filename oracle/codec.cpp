// Oracle for the 12 Hz codec decoder (codes -> 24 kHz waveform) -- TEST
// INFRASTRUCTURE ONLY.
//
// A plain, slow fp64 CPU restatement of what the decoder computes for one
// window of frames decoded from a zero state.  Only tests/, the smoke check
// and the benchmark's CPU-baseline leg may load it; it shares no code, header
// or table with the CUDA library.
//
// Sources followed (page title, section):
//  * "Qwen3-TTS 移植 ncnn 简明教程" (ncnn discussion 6798), section 1
//    "先搞清楚结构", Codec Decoder bullet: SplitRVQ dequantisation (16
//    codebooks of 2048 x 256) -> 8-layer transformer with a sliding window of
//    72 (hidden 512, head_dim 64, RoPE theta 1e4, LayerScale) -> 2 x
//    (transposed convolution + ConvNeXt) -> DAC-style vocoder (SnakeBeta
//    activations, upsampling [8, 5, 4, 3]) -> x1920 samples per frame at
//    24 kHz; one feed-forward pass.  Section 3/4: SnakeBeta keeps exp(alpha)
//    and exp(beta) of log-scale parameters.
//  * Mizuoto "Qwen3-TTS" engine page, section "速度": the decoder is causal
//    from end to end, and a request is decoded on a grid of 300-frame chunks
//    with 25 frames of left context (the chunk grid lives in the tests).
//
// Readings where the pages are silent (each also listed with the design notes):
//  * SplitRVQ: codebook 0 (semantic) and codebooks 1..15 (acoustic) are two
//    residual quantisers; each sums its codebook rows and has its own output
//    projection 256 -> 512 without bias; the two projections are added.
//  * transformer layer: pre-norm RMSNorm (eps 1e-5), q/k/v/o projections
//    without bias, 8 heads of 64, rotate-half RoPE at the frame's index in
//    the window, causal attention over the last 72 frames (t-71..t), a SiLU-
//    gated MLP of width 1024; LayerScale multiplies each residual branch by a
//    per-channel vector before it is added; a final RMSNorm.
//  * upsampling stage: transposed convolution with kernel = stride = 2
//    (512 -> 512 channels, bias), then a ConvNeXt block: causal depthwise
//    convolution of width 7 (bias), LayerNorm over channels (eps 1e-6,
//    weight and bias), Linear 512 -> 2048 (bias), exact-erf GELU, Linear
//    2048 -> 512 (bias), per-channel scale gamma, residual.
//  * DAC vocoder: causal Conv1d 512 -> 1536 (k 7) and four blocks halving the
//    channels (1536 -> 768 -> 384 -> 192 -> 96) with strides 8, 5, 4, 3:
//    SnakeBeta, causal transposed convolution (kernel 2 x stride, the
//    trailing `stride` samples of the full output dropped), three residual
//    units with dilations 1, 3, 9 (SnakeBeta, Conv k 7 dilated, SnakeBeta,
//    Conv k 1, added to the input); then SnakeBeta, Conv1d 96 -> 1 (k 7) and
//    tanh.  SnakeBeta(x) = x + sin^2(exp(a) x) / (exp(b) + 1e-9) per channel.
//  * causal convolution: y[t] = b + sum_k W[k] x[t - (K-1-k) d], zeros
//    before the window's first frame.
//
// Weight layouts (shared with the library's ABI, read here by their
// definitions): Linear [out][in]; Conv1d [Cout][K][Cin] (tap k multiplies
// x[t - (K-1-k) d]); depthwise [C][7]; transposed convolution
// [stride][Cout][K/stride][Cin], element (r, co, j, ci) = kernel tap
// k = r + j * stride of input channel ci to output channel co.
//
// Numerics: all arithmetic in fp64 on the weight values handed in (fp32, or
// bf16-exact values for a bf16 model).  Parity of the waveform for random
// weights is unpinned beyond the invariants the tests check (the pages print
// no decoder outputs).
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include <algorithm>

extern "C" {

typedef struct {
    int n_codebooks, codebook_size, codebook_dim;   // 16, 2048, 256
    int hidden, n_layers, n_heads, head_dim, ffn;   // 512, 8, 8, 64, 1024
    int window;                                     // 72
    float rope_theta, rms_eps, ln_eps;              // 1e4, 1e-5, 1e-6
    int n_up, up_ffn;                               // 2 upsampling stages, ConvNeXt width 2048
    int dac_channels;                               // 1536
    int n_blocks;                                   // 4
    int strides[4];                                 // 8, 5, 4, 3
} oc_config;

typedef struct {
    const float* codebooks;   // [16][2048][256]
    const float* proj_sem;    // [512][256]
    const float* proj_ac;     // [512][256]
    // transformer, per layer (stacked over layers)
    const float* attn_norm;   // [L][512]
    const float* wqkv;        // [L][3*512][512]  rows: q, k, v
    const float* wo;          // [L][512][512]
    const float* ls_attn;     // [L][512]
    const float* mlp_norm;    // [L][512]
    const float* wgu;         // [L][2*F][512]    rows: gate, up
    const float* wd;          // [L][512][F]
    const float* ls_mlp;      // [L][512]
    const float* final_norm;  // [512]
    // upsampling stages (stacked over stages)
    const float* up_w;        // [U][2][512][1][512]
    const float* up_b;        // [U][512]
    const float* dw_w;        // [U][512][7]
    const float* dw_b;        // [U][512]
    const float* ln_w;        // [U][512]
    const float* ln_b;        // [U][512]
    const float* fc1_w;       // [U][2048][512]
    const float* fc1_b;       // [U][2048]
    const float* fc2_w;       // [U][512][2048]
    const float* fc2_b;       // [U][512]
    const float* gamma;       // [U][512]
    // vocoder
    const float* in_w;        // [1536][7][512]
    const float* in_b;        // [1536]
    const float* blk[4][4];   // per block: snake a, b [Cin]; transposed conv [s][Cout][2][Cin], bias [Cout]
    const float* unit[4][3][8];  // per block and residual unit: snake a1, b1 [Cout], conv w1 [Cout][7][Cout],
                                 // c1 [Cout], snake a2, b2 [Cout], conv w2 [Cout][1][Cout], c2 [Cout]
    const float* out_a;       // [96]
    const float* out_b;       // [96]
    const float* out_w;       // [1][7][96]
    const float* out_bias;    // [1]
} oc_weights;

}  // extern "C"

namespace {

using Mat = std::vector<double>;   // [T][C], channels last

// ---- building blocks (each the plain definition) ----

void rmsnorm(const double* x, int n, const float* w, double eps, double* y) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    const double r = 1.0 / std::sqrt(ss / n + eps);
    for (int i = 0; i < n; ++i) y[i] = x[i] * r * (double)w[i];
}

void layernorm(const double* x, int n, const float* w, const float* b, double eps, double* y) {
    double mu = 0.0;
    for (int i = 0; i < n; ++i) mu += x[i];
    mu /= n;
    double var = 0.0;
    for (int i = 0; i < n; ++i) var += (x[i] - mu) * (x[i] - mu);
    var /= n;
    const double r = 1.0 / std::sqrt(var + eps);
    for (int i = 0; i < n; ++i) y[i] = (x[i] - mu) * r * (double)w[i] + (double)b[i];
}

// y[o] = sum_i W[o][i] x[i] (+ bias)
void linear(const float* W, const float* bias, int out, int in, const double* x, double* y) {
    for (int o = 0; o < out; ++o) {
        double acc = bias ? (double)bias[o] : 0.0;
        const float* w = W + (size_t)o * in;
        for (int i = 0; i < in; ++i) acc += (double)w[i] * x[i];
        y[o] = acc;
    }
}

double gelu(double v) { return 0.5 * v * (1.0 + std::erf(v / std::sqrt(2.0))); }
double silu(double v) { return v / (1.0 + std::exp(-v)); }

// SnakeBeta, log-scale parameters: x + sin^2(e^a x) / (e^b + 1e-9)
void snake(Mat& x, int T, int C, const float* la, const float* lb) {
    for (int c = 0; c < C; ++c) {
        const double a = std::exp((double)la[c]), ib = 1.0 / (std::exp((double)lb[c]) + 1e-9);
        for (int t = 0; t < T; ++t) {
            double& v = x[(size_t)t * C + c];
            const double s = std::sin(a * v);
            v = v + ib * s * s;
        }
    }
}

// causal Conv1d: y[t][co] = b[co] + sum_{k, ci} W[co][k][ci] x[t - (K-1-k) d][ci]
Mat conv1d(const Mat& x, int T, int Cin, int Cout, int K, int d, const float* W, const float* b) {
    Mat y((size_t)T * Cout);
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t)
        for (int co = 0; co < Cout; ++co) {
            double acc = b ? (double)b[co] : 0.0;
            for (int k = 0; k < K; ++k) {
                const int ts = t - (K - 1 - k) * d;
                if (ts < 0) continue;
                const float* w = W + ((size_t)co * K + k) * Cin;
                const double* xs = &x[(size_t)ts * Cin];
                for (int ci = 0; ci < Cin; ++ci) acc += (double)w[ci] * xs[ci];
            }
            y[(size_t)t * Cout + co] = acc;
        }
    return y;
}

// causal transposed convolution, stride s, kernel Kt (a multiple of s):
// input frame m adds W(k, co, ci) x[m][ci] to output sample m*s + k for
// k < Kt; the full output has (T-1) s + Kt samples, of which the first T*s
// are kept.  W(k, co, ci) is element (k mod s, co, k div s, ci) of the stored
// [s][Cout][Kt/s][Cin] array.
Mat conv_transpose(const Mat& x, int T, int Cin, int Cout, int s, int Kt, const float* W, const float* b) {
    const int J = Kt / s;
    const int n_full = (T - 1) * s + Kt;
    Mat full((size_t)n_full * Cout, 0.0);
    // output sample m*s + k gets input m's contribution; parallel over the
    // residue class of k so no two threads add into the same sample
    for (int m = 0; m < T; ++m)
#pragma omp parallel for schedule(static)
        for (int k = 0; k < Kt; ++k) {
            const int r = k % s, j = k / s;
            for (int co = 0; co < Cout; ++co) {
                const float* w = W + (((size_t)r * Cout + co) * J + j) * Cin;
                double acc = 0.0;
                for (int ci = 0; ci < Cin; ++ci) acc += (double)w[ci] * x[(size_t)m * Cin + ci];
                full[(size_t)(m * s + k) * Cout + co] += acc;
            }
        }
    Mat y((size_t)T * s * Cout);
    for (int n = 0; n < T * s; ++n)
        for (int co = 0; co < Cout; ++co) y[(size_t)n * Cout + co] = full[(size_t)n * Cout + co] + (b ? (double)b[co] : 0.0);
    return y;
}

// rotate-half RoPE on one head vector at position pos
void rope(double* v, int hd, int pos, double theta) {
    const int h = hd / 2;
    for (int j = 0; j < h; ++j) {
        const double f = std::pow(theta, -2.0 * j / hd);
        const double ang = pos * f;
        const double c = std::cos(ang), sn = std::sin(ang);
        const double a = v[j], b = v[j + h];
        v[j] = a * c - b * sn;
        v[j + h] = b * c + a * sn;
    }
}

}  // namespace

extern "C" {

// Causal sliding-window multi-head attention over one window: q, k, v [T][H*hd]
// (RoPE already applied); query t attends to frames max(0, t-W+1)..t.
void oracle_codec_attention(const double* q, const double* k, const double* v, int T, int H, int hd, int W,
                            double* out) {
    const double scale = 1.0 / std::sqrt((double)hd);
    std::vector<double> p(T);
    for (int h = 0; h < H; ++h)
        for (int t = 0; t < T; ++t) {
            const int s0 = std::max(0, t - W + 1);
            double mx = -INFINITY;
            for (int s = s0; s <= t; ++s) {
                double d = 0.0;
                for (int i = 0; i < hd; ++i) d += q[(size_t)t * H * hd + h * hd + i] * k[(size_t)s * H * hd + h * hd + i];
                p[s] = d * scale;
                mx = std::max(mx, p[s]);
            }
            double z = 0.0;
            for (int s = s0; s <= t; ++s) { p[s] = std::exp(p[s] - mx); z += p[s]; }
            for (int i = 0; i < hd; ++i) {
                double acc = 0.0;
                for (int s = s0; s <= t; ++s) acc += p[s] * v[(size_t)s * H * hd + h * hd + i];
                out[(size_t)t * H * hd + h * hd + i] = acc / z;
            }
        }
}

void oracle_codec_conv1d(const double* x, int T, int Cin, int Cout, int K, int d, const float* W, const float* b,
                         double* y) {
    Mat xx(x, x + (size_t)T * Cin);
    Mat r = conv1d(xx, T, Cin, Cout, K, d, W, b);
    std::memcpy(y, r.data(), r.size() * sizeof(double));
}

void oracle_codec_conv_transpose(const double* x, int T, int Cin, int Cout, int s, int Kt, const float* W,
                                 const float* b, double* y) {
    Mat xx(x, x + (size_t)T * Cin);
    Mat r = conv_transpose(xx, T, Cin, Cout, s, Kt, W, b);
    std::memcpy(y, r.data(), r.size() * sizeof(double));
}

void oracle_codec_snake(double* x, int T, int C, const float* la, const float* lb) {
    Mat xx(x, x + (size_t)T * C);
    snake(xx, T, C, la, lb);
    std::memcpy(x, xx.data(), xx.size() * sizeof(double));
}

// One window of T frames decoded from a zero state.  codes [T][16] (codebook 0
// first); latent_out (optional) [T][512] after the transformer's final norm;
// wav [T * 1920 (product of the strides x 4)].  Returns 0, or 1 for a bad
// argument (a code outside the codebook).
int oracle_codec_decode(const oc_config* c, const oc_weights* w, const int32_t* codes, int T, double* latent_out,
                        double* wav) {
    const int D = c->hidden, Dc = c->codebook_dim, V = c->codebook_size, NQ = c->n_codebooks;
    const int H = c->n_heads, hd = c->head_dim, F = c->ffn, L = c->n_layers;
    for (int i = 0; i < T * NQ; ++i)
        if (codes[i] < 0 || codes[i] >= V) return 1;
    if (T <= 0) return 0;
    // SplitRVQ dequantisation
    Mat x((size_t)T * D);
    {
        std::vector<double> zs(Dc), za(Dc), ys(D), ya(D);
        for (int t = 0; t < T; ++t) {
            for (int i = 0; i < Dc; ++i) { zs[i] = 0.0; za[i] = 0.0; }
            for (int q = 0; q < NQ; ++q) {
                const float* e = w->codebooks + ((size_t)q * V + codes[t * NQ + q]) * Dc;
                std::vector<double>& z = q == 0 ? zs : za;
                for (int i = 0; i < Dc; ++i) z[i] += (double)e[i];
            }
            linear(w->proj_sem, nullptr, D, Dc, zs.data(), ys.data());
            linear(w->proj_ac, nullptr, D, Dc, za.data(), ya.data());
            for (int i = 0; i < D; ++i) x[(size_t)t * D + i] = ys[i] + ya[i];
        }
    }
    // transformer
    {
        std::vector<double> hbuf(D), q((size_t)T * D), k((size_t)T * D), v((size_t)T * D), o((size_t)T * D),
            qkv(3 * D), tmp(D), gu(2 * F), a(F);
        for (int l = 0; l < L; ++l) {
            const float* wqkv = w->wqkv + (size_t)l * 3 * D * D;
            for (int t = 0; t < T; ++t) {
                rmsnorm(&x[(size_t)t * D], D, w->attn_norm + (size_t)l * D, c->rms_eps, hbuf.data());
                linear(wqkv, nullptr, 3 * D, D, hbuf.data(), qkv.data());
                for (int i = 0; i < D; ++i) {
                    q[(size_t)t * D + i] = qkv[i];
                    k[(size_t)t * D + i] = qkv[D + i];
                    v[(size_t)t * D + i] = qkv[2 * D + i];
                }
                for (int h = 0; h < H; ++h) {
                    rope(&q[(size_t)t * D + h * hd], hd, t, c->rope_theta);
                    rope(&k[(size_t)t * D + h * hd], hd, t, c->rope_theta);
                }
            }
            oracle_codec_attention(q.data(), k.data(), v.data(), T, H, hd, c->window, o.data());
            for (int t = 0; t < T; ++t) {
                linear(w->wo + (size_t)l * D * D, nullptr, D, D, &o[(size_t)t * D], tmp.data());
                for (int i = 0; i < D; ++i) x[(size_t)t * D + i] += (double)w->ls_attn[(size_t)l * D + i] * tmp[i];
                rmsnorm(&x[(size_t)t * D], D, w->mlp_norm + (size_t)l * D, c->rms_eps, hbuf.data());
                linear(w->wgu + (size_t)l * 2 * F * D, nullptr, 2 * F, D, hbuf.data(), gu.data());
                for (int i = 0; i < F; ++i) a[i] = silu(gu[i]) * gu[F + i];
                linear(w->wd + (size_t)l * D * F, nullptr, D, F, a.data(), tmp.data());
                for (int i = 0; i < D; ++i) x[(size_t)t * D + i] += (double)w->ls_mlp[(size_t)l * D + i] * tmp[i];
            }
        }
        for (int t = 0; t < T; ++t) {
            rmsnorm(&x[(size_t)t * D], D, w->final_norm, c->rms_eps, hbuf.data());
            for (int i = 0; i < D; ++i) x[(size_t)t * D + i] = hbuf[i];
        }
        if (latent_out) std::memcpy(latent_out, x.data(), x.size() * sizeof(double));
    }
    // upsampling: transposed convolution x2, then ConvNeXt
    int n = T;
    for (int u = 0; u < c->n_up; ++u) {
        x = conv_transpose(x, n, D, D, 2, 2, w->up_w + (size_t)u * 2 * D * D, w->up_b + (size_t)u * D);
        n *= 2;
        const int F2 = c->up_ffn;
        const float* dw = w->dw_w + (size_t)u * D * 7;
        std::vector<double> dcv(D), nn(D), h1(F2), h2(D);
        Mat res = x;
        for (int t = 0; t < n; ++t) {
            for (int ch = 0; ch < D; ++ch) {
                double acc = (double)w->dw_b[(size_t)u * D + ch];
                for (int kk = 0; kk < 7; ++kk) {
                    const int ts = t - (6 - kk);
                    if (ts >= 0) acc += (double)dw[ch * 7 + kk] * res[(size_t)ts * D + ch];
                }
                dcv[ch] = acc;
            }
            layernorm(dcv.data(), D, w->ln_w + (size_t)u * D, w->ln_b + (size_t)u * D, c->ln_eps, nn.data());
            linear(w->fc1_w + (size_t)u * F2 * D, w->fc1_b + (size_t)u * F2, F2, D, nn.data(), h1.data());
            for (int i = 0; i < F2; ++i) h1[i] = gelu(h1[i]);
            linear(w->fc2_w + (size_t)u * D * F2, w->fc2_b + (size_t)u * D, D, F2, h1.data(), h2.data());
            for (int ch = 0; ch < D; ++ch) x[(size_t)t * D + ch] = res[(size_t)t * D + ch] + (double)w->gamma[(size_t)u * D + ch] * h2[ch];
        }
    }
    // DAC-style vocoder
    int C = c->dac_channels;
    x = conv1d(x, n, D, C, 7, 1, w->in_w, w->in_b);
    for (int b = 0; b < c->n_blocks; ++b) {
        const int s = c->strides[b], Co = C / 2;
        snake(x, n, C, w->blk[b][0], w->blk[b][1]);
        x = conv_transpose(x, n, C, Co, s, 2 * s, w->blk[b][2], w->blk[b][3]);
        n *= s;
        C = Co;
        static const int dil[3] = {1, 3, 9};
        for (int u = 0; u < 3; ++u) {
            const float* const* p = w->unit[b][u];
            Mat r = x;
            snake(r, n, C, p[0], p[1]);
            r = conv1d(r, n, C, C, 7, dil[u], p[2], p[3]);
            snake(r, n, C, p[4], p[5]);
            r = conv1d(r, n, C, C, 1, 1, p[6], p[7]);
            for (size_t i = 0; i < x.size(); ++i) x[i] += r[i];
        }
    }
    snake(x, n, C, w->out_a, w->out_b);
    Mat y = conv1d(x, n, C, 1, 7, 1, w->out_w, w->out_bias);
    for (int i = 0; i < n; ++i) wav[i] = std::tanh(y[i]);
    return 0;
}

}  // extern "C"
