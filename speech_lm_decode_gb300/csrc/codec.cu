// 12 Hz codec decoder on the GPU: codes -> 24 kHz waveform (q3codec.h).
//
// The structure follows the Codec Decoder bullet of "Qwen3-TTS 移植 ncnn 简明
// 教程" (ncnn discussion 6798, section 1) and the chunk grid and streaming
// schedule of the Mizuoto "Qwen3-TTS" page (section "速度"); the readings
// where those pages are silent are stated in q3codec.h.
//
// Activations are fp32 and channels-last ([frames or samples][channels]).
// Every product with a weight matrix is a projection on the library's GEMM
// path (tcgen05 tensor cores from tc_min_tokens rows, with the fp32 operand
// as bf16 high + low parts; GEMV / tiled CUDA-core kernels below that):
//   * a causal convolution of width K and dilation d is one GEMM over an
//     im2col operand whose row t is [x[t-(K-1)d], ..., x[t]] (K x Cin), with
//     the weight [Cout][K][Cin] as the matrix;
//   * a causal transposed convolution with kernel 2s and stride s is one GEMM
//     whose row m is [x[m], x[m-1]] and whose s * Cout outputs are samples
//     m*s + r, r < s, of every output channel (the weight [s][Cout][2][Cin] as
//     the matrix), so its output is already channels-last [M * s][Cout];
//   * SnakeBeta is applied while the operand is gathered (snake(0) = 0, so
//     the zero padding commutes with it).
// The operand kernels write the tensor-core operand (bf16 high / low parts)
// directly when the product runs there.  Small kernels: dequantisation
// gather, RoPE, window attention, depthwise conv + LayerNorm, GELU,
// LayerScale / gamma residual adds, and the single-channel output
// convolution with tanh.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "pdl.cuh"
#include "q3codec.h"

using namespace q3;

namespace {

constexpr int CHUNK = 300;     // frames per chunk of a request's grid
constexpr int CONTEXT = 25;    // left-context frames decoded before a chunk
constexpr int S_FIRST = 4;     // frames before the first streamed decode
constexpr int S_EVERY = 12;    // frames between later streamed decodes
constexpr size_t ALIGN = 256;

// ------------------------------------------------------------------ kernels
// SnakeBeta of value v with the channel's (exp(a), 1 / (exp(b) + 1e-9))
__device__ __forceinline__ float snake(float v, float2 ab) {
    const float s = sinf(ab.x * v);
    return fmaf(ab.y * s, s, v);
}

// (exp(a), 1 / (exp(b) + 1e-9)) per channel, from the log-scale parameters
__global__ void snake_table_kernel(const float* __restrict__ la, const float* __restrict__ lb, int C,
                                   float2* __restrict__ out) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c < C) out[c] = make_float2(expf(la[c]), 1.0f / (expf(lb[c]) + 1e-9f));
}

// bias [C] repeated s times: the per-output bias of a transposed convolution's GEMM
__global__ void repeat_kernel(const float* __restrict__ b, int C, int s, float* __restrict__ out) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < C * s) out[i] = b[i % C];
}

// SplitRVQ: zs[t] = cb[0][c_0], za[t] = sum_{q >= 1} cb[q][c_q]; a code out of
// range sets the BOUNDS bit and reads row 0
template <typename T>
__global__ void dequant_kernel(const int32_t* __restrict__ codes, int NQ, int V, int Dc, const T* __restrict__ cb,
                               float* __restrict__ zs, float* __restrict__ za, int* __restrict__ err) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    __shared__ int cs[32];
    if (threadIdx.x < NQ) {
        int c = codes[(size_t)t * NQ + threadIdx.x];
        if (c < 0 || c >= V) { atomicOr(err, ERRB_BOUNDS); c = 0; }
        cs[threadIdx.x] = c;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < Dc; i += blockDim.x) {
        zs[(size_t)t * Dc + i] = to_f(cb[(size_t)cs[0] * Dc + i]);
        float a = 0.f;
        for (int q = 1; q < NQ; ++q) a += to_f(cb[((size_t)q * V + cs[q]) * Dc + i]);
        za[(size_t)t * Dc + i] = a;
    }
}

// rotate-half RoPE on q and k of qkv [T][3D] at the frame index (head_dim 64)
__global__ void rope64_kernel(float* __restrict__ qkv, int D, float theta) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    const int H = D / 64;
    for (int i = threadIdx.x; i < 2 * H * 32; i += blockDim.x) {
        const int which = i / (H * 32), h = (i / 32) % H, j = i % 32;
        float* v = qkv + (size_t)t * 3 * D + which * D + h * 64;
        const float f = powf(theta, -2.0f * j / 64.0f);
        float sn, cs;
        sincosf((float)t * f, &sn, &cs);
        const float a = v[j], b = v[j + 32];
        v[j] = a * cs - b * sn;
        v[j + 32] = b * cs + a * sn;
    }
}

// causal window attention, one (frame, head) per block of 128 threads
__global__ void __launch_bounds__(128) window_attn_kernel(const float* __restrict__ qkv, int D, int W,
                                                          float* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x, h = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int s0 = max(0, t - W + 1), n = t - s0 + 1;
    extern __shared__ float sc[];   // [n]
    __shared__ float red[2];
    const float* q = qkv + (size_t)t * 3 * D + h * 64;
    const float q0 = q[lane] * 0.125f, q1 = q[lane + 32] * 0.125f;   // 1/sqrt(64)
    for (int j = warp; j < n; j += 4) {
        const float* k = qkv + (size_t)(s0 + j) * 3 * D + D + h * 64;
        const float d = warp_sum(fmaf(q0, k[lane], q1 * k[lane + 32]));
        if (lane == 0) sc[j] = d;
    }
    __syncthreads();
    if (warp == 0) {
        float mx = -INFINITY;
        for (int j = lane; j < n; j += 32) mx = fmaxf(mx, sc[j]);
        mx = warp_max(mx);
        float z = 0.f;
        for (int j = lane; j < n; j += 32) { const float p = expf(sc[j] - mx); sc[j] = p; z += p; }
        z = warp_sum(z);
        if (lane == 0) red[0] = z;
    }
    __syncthreads();
    if (threadIdx.x < 64) {
        float acc = 0.f;
        for (int j = 0; j < n; ++j) acc = fmaf(sc[j], qkv[(size_t)(s0 + j) * 3 * D + 2 * D + h * 64 + threadIdx.x], acc);
        out[(size_t)t * D + h * 64 + threadIdx.x] = acc / red[0];
    }
}

// x[m][c] += g[c] * y[m][c]
__global__ void scale_add_kernel(float* __restrict__ x, const float* __restrict__ y, const float* __restrict__ g,
                                 size_t n, int C) {
    pdl_wait();
    pdl_trigger();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        x[i] = fmaf(g[i % C], y[i], x[i]);
}

// ConvNeXt front: causal depthwise conv (width 7) then LayerNorm over the
// channels, one frame per block; output fp32 [T][C] or the bf16 parts
__global__ void __launch_bounds__(256) dwconv_ln_kernel(const float* __restrict__ x, int C,
                                                        const float* __restrict__ w, const float* __restrict__ b,
                                                        const float* __restrict__ lw, const float* __restrict__ lb,
                                                        float eps, float* __restrict__ out, bf16* __restrict__ hi,
                                                        bf16* __restrict__ lo) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    extern __shared__ float dv[];   // [C]
    __shared__ float red[8];
    float s = 0.f;
    for (int c = threadIdx.x; c < C; c += 256) {
        float acc = b[c];
        for (int k = 0; k < 7; ++k) {
            const int ts = t - 6 + k;
            if (ts >= 0) acc = fmaf(w[c * 7 + k], x[(size_t)ts * C + c], acc);
        }
        dv[c] = acc;
        s += acc;
    }
    auto block_sum = [&](float v) {
        v = warp_sum(v);
        __syncthreads();
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
        __syncthreads();
        float r = 0.f;
        for (int i = 0; i < 8; ++i) r += red[i];
        return r;
    };
    const float mu = block_sum(s) / C;
    float v2 = 0.f;
    for (int c = threadIdx.x; c < C; c += 256) { const float d = dv[c] - mu; v2 = fmaf(d, d, v2); }
    const float r = rsqrtf(block_sum(v2) / C + eps);
    for (int c = threadIdx.x; c < C; c += 256) {
        const float y = fmaf((dv[c] - mu) * r, lw[c], lb[c]);
        if (hi) {
            const bf16 hv = __float2bfloat16_rn(y);
            hi[(size_t)t * C + c] = hv;
            lo[(size_t)t * C + c] = __float2bfloat16_rn(y - __bfloat162float(hv));
        } else {
            out[(size_t)t * C + c] = y;
        }
    }
}

// exact GELU of h, written as fp32 (in place allowed) or as the bf16 parts
__global__ void gelu_kernel(const float* h, size_t n, float* out, bf16* __restrict__ hi,
                            bf16* __restrict__ lo) {
    pdl_wait();
    pdl_trigger();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const float v = h[i];
        const float y = 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
        if (hi) {
            const bf16 hv = __float2bfloat16_rn(y);
            hi[i] = hv;
            lo[i] = __float2bfloat16_rn(y - __bfloat162float(hv));
        } else {
            out[i] = y;
        }
    }
}

// Operand of a convolution as a GEMM: row m, column (k, ci) =
// snake(x[m - lag(k)][ci]) (0 before the first row), lag(k) = (K-1-k) d for a
// causal convolution, k for the transposed convolution's [x[m], x[m-1]].
// Four channels per thread (Cin % 4 == 0).
__global__ void gather_kernel(const float* __restrict__ x, int M, int Cin, int K, int d, int rev,
                              const float2* __restrict__ ab, float* __restrict__ out, bf16* __restrict__ hi,
                              bf16* __restrict__ lo) {
    pdl_wait();
    pdl_trigger();
    const int C4 = Cin >> 2;
    const size_t per_row = (size_t)K * C4;
    const size_t n = (size_t)M * per_row;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int m = (int)(i / per_row);
        const int rem = (int)(i - (size_t)m * per_row);
        const int k = rem / C4, c = (rem - k * C4) * 4;
        const int src = m - (rev ? k : (K - 1 - k) * d);
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (src >= 0) {
            v = *reinterpret_cast<const float4*>(x + (size_t)src * Cin + c);
            if (ab) {
                v.x = snake(v.x, ab[c]); v.y = snake(v.y, ab[c + 1]);
                v.z = snake(v.z, ab[c + 2]); v.w = snake(v.w, ab[c + 3]);
            }
        }
        const size_t o = (size_t)m * K * Cin + (size_t)k * Cin + c;
        if (hi) {
            const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bf16 hv = __float2bfloat16_rn(vv[j]);
                hi[o + j] = hv;
                lo[o + j] = __float2bfloat16_rn(vv[j] - __bfloat162float(hv));
            }
        } else {
            *reinterpret_cast<float4*>(out + o) = v;
        }
    }
}

// output convolution to one channel (width 7) after SnakeBeta, then tanh; one
// warp per sample, lanes over the channels
template <typename T>
__global__ void out_conv_kernel(const float* __restrict__ x, int M, int C, const float2* __restrict__ ab,
                                const T* __restrict__ w, const float* __restrict__ b, float* __restrict__ wav) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int m = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (m >= M) return;
    float acc = 0.f;
    for (int k = 0; k < 7; ++k) {
        const int src = m - 6 + k;
        if (src < 0) continue;
        for (int c = lane; c < C; c += 32) acc = fmaf(to_f(w[k * C + c]), snake(x[(size_t)src * C + c], ab[c]), acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) wav[m] = tanhf(acc + b[0]);
}

unsigned grid_for(size_t n, int threads) {
    const size_t g = (n + threads - 1) / threads;
    return (unsigned)std::min<size_t>(g, (size_t)device_sm_count() * 32);
}

}  // namespace

// ------------------------------------------------------------------ handle
struct q3codec {
    q3codec_config c{};
    q3codec_weights w{};
    char* ws = nullptr;
    cudaStream_t st = nullptr;
    std::string last_error;
    int spf = 0;
    // workspace regions (byte offsets)
    size_t codes, zs, za, x, qkv, att, tmp, op, act, bufA, bufB, bufR, col, tcs, snk, rep, wav, err, total;
    size_t tc_bytes = 0, col_elems = 0, buf_elems = 0, r_elems = 0, wav_elems = 0;
    size_t snk_blk[Q3C_MAX_BLOCKS], snk_unit[Q3C_MAX_BLOCKS][3][2], snk_out;   // float2 offsets into snk
    size_t rep_up[2], rep_blk[Q3C_MAX_BLOCKS];                                  // float offsets into rep
    int up_cnt = 0;
    // streaming state
    std::vector<int32_t> s_codes;
    long s_sent = 0;      // samples sent
    int s_due = S_FIRST;
    bool s_final = false;
    int kernels = 0;      // launches of the last window

    template <typename T> T* p(size_t off) const { return reinterpret_cast<T*>(ws + off); }
    TcScratch tc() const {
        TcScratch t;
        t.base = c.dtype == Q3_BF16 ? p<void>(tcs) : nullptr;
        t.bytes = c.dtype == Q3_BF16 ? tc_bytes : 0;
        t.min_tokens = c.tc_min_tokens == 0 ? 16 : c.tc_min_tokens;
        return t;
    }
    int* errp() const { return p<int>(err); }
};

namespace {

int cfail(q3codec* h, int code, const char* fmt, ...) {
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

#define CC(call)                                                                                     \
    do {                                                                                             \
        cudaError_t e_ = (call);                                                                     \
        if (e_ != cudaSuccess) return cfail(h, Q3_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
    } while (0)

bool cfg_ok(const q3codec_config* c, std::string* why) {
    auto bad = [&](const char* m) { if (why) *why = m; return false; };
    if (!c) return bad("config is NULL");
    if (c->dtype != Q3_F32 && c->dtype != Q3_BF16) return bad("dtype must be Q3_F32 or Q3_BF16");
    if (c->n_codebooks < 2 || c->n_codebooks > 32) return bad("n_codebooks must be 2..32");
    if (c->codebook_size < 1 || c->codebook_dim < 8 || c->codebook_dim % 8) return bad("bad codebook shape");
    if (c->head_dim != 64) return bad("head_dim must be 64");
    if (c->n_heads < 1 || c->hidden != c->n_heads * 64) return bad("hidden must be n_heads x 64");
    if (c->n_layers < 0 || c->ffn < 8 || c->ffn % 8 || c->window < 1) return bad("bad transformer shape");
    if (c->n_up < 0 || c->n_up > 2) return bad("n_up must be 0..2");
    if (c->up_ffn < 8 || c->up_ffn % 8) return bad("up_ffn must be a positive multiple of 8");
    if (c->n_blocks < 1 || c->n_blocks > Q3C_MAX_BLOCKS) return bad("n_blocks must be 1..4");
    if (c->dac_channels < 8 || c->dac_channels % (8 << c->n_blocks)) return bad("dac_channels must stay a multiple of 8 when halved per block");
    for (int b = 0; b < c->n_blocks; ++b)
        if (c->strides[b] < 1 || c->strides[b] > 16) return bad("strides must be 1..16");
    if (c->max_frames < 1 || c->max_frames > 4096) return bad("max_frames must be 1..4096");
    if (!(c->rms_eps > 0.f) || !(c->ln_eps > 0.f) || !(c->rope_theta > 0.f)) return bad("eps and theta must be positive");
    return true;
}

// widths and lengths of every stage, and the workspace regions
void layout(q3codec* h) {
    const q3codec_config& c = h->c;
    const size_t T = (size_t)c.max_frames, D = c.hidden, F = c.ffn, F2 = c.up_ffn, Dc = c.codebook_dim;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off += (bytes + ALIGN - 1) / ALIGN * ALIGN; return o; };
    // stage sizes
    size_t buf = T * std::max(D * 3, F);              // transformer scratch fits in bufA / bufB too
    size_t maxK = std::max({Dc, D, F, F2, (size_t)7 * D}), maxMK = T * std::max({Dc, D, F});
    size_t n = T;
    for (int u = 0; u < c.n_up; ++u) {
        n *= 2;
        buf = std::max(buf, n * std::max(D, F2));
        maxMK = std::max(maxMK, n * std::max(D, F2));
    }
    size_t C = c.dac_channels, r = 0;
    buf = std::max(buf, n * C);
    maxMK = std::max(maxMK, n * 7 * D);
    for (int b = 0; b < c.n_blocks; ++b) {
        const size_t s = c.strides[b], Co = C / 2;
        maxK = std::max({maxK, 2 * C, 7 * Co});
        maxMK = std::max(maxMK, n * 2 * C);
        n *= s;
        C = Co;
        buf = std::max(buf, n * C);
        r = std::max(r, n * C);
        maxMK = std::max(maxMK, n * 7 * C);
    }
    h->buf_elems = buf;
    h->r_elems = r;
    h->wav_elems = n;
    h->spf = (int)(n / T);
    // fp32 operand rows of products on the CUDA cores: fewer than tc_min_tokens
    // rows on the tensor-core path, every product without it
    const int tmin = c.tc_min_tokens == 0 ? 16 : c.tc_min_tokens;
    h->col_elems = (c.dtype == Q3_BF16 && tmin > 0) ? (size_t)tmin * maxK : maxMK;
    h->tc_bytes = c.dtype == Q3_BF16 ? maxMK * 4 : 0;  // bf16 high + low parts
    h->codes = take(T * c.n_codebooks * 4);
    h->zs = take(T * Dc * 4);
    h->za = take(T * Dc * 4);
    h->x = take(T * D * 4);
    h->qkv = take(T * 3 * D * 4);
    h->att = take(T * D * 4);
    h->tmp = take(T * D * 4);
    h->op = take(T * std::max(D, F) * 4);
    h->act = take(T * F * 4);
    h->bufA = take(buf * 4);
    h->bufB = take(buf * 4);
    h->bufR = take(std::max<size_t>(r, 1) * 4);
    h->col = take(std::max(h->col_elems, h->buf_elems) * 4);
    h->tcs = take(std::max<size_t>(h->tc_bytes, 256));
    // SnakeBeta tables
    size_t nsk = 0;
    C = c.dac_channels;
    for (int b = 0; b < c.n_blocks; ++b) {
        h->snk_blk[b] = nsk; nsk += C;
        const size_t Co = C / 2;
        for (int u = 0; u < 3; ++u) { h->snk_unit[b][u][0] = nsk; nsk += Co; h->snk_unit[b][u][1] = nsk; nsk += Co; }
        C = Co;
    }
    h->snk_out = nsk; nsk += C;
    h->snk = take(nsk * sizeof(float2));
    size_t nrep = 0;
    for (int u = 0; u < c.n_up; ++u) { h->rep_up[u] = nrep; nrep += 2 * D; }
    C = c.dac_channels;
    for (int b = 0; b < c.n_blocks; ++b) { h->rep_blk[b] = nrep; nrep += (size_t)c.strides[b] * (C / 2); C /= 2; }
    h->rep = take(std::max<size_t>(nrep, 1) * 4);
    h->wav = take(n * 4);
    h->err = take(16);
    h->total = off;
}

size_t esz(int dtype) { return dtype == Q3_BF16 ? 2 : 4; }

bool is_dev(const void* p) {
    cudaPointerAttributes pa;
    const bool d = cudaPointerGetAttributes(&pa, p) == cudaSuccess &&
                   (pa.type == cudaMemoryTypeDevice || pa.type == cudaMemoryTypeManaged);
    cudaGetLastError();
    return d;
}

// ------------------------------------------------------------------ one window
class Window {
public:
    explicit Window(q3codec* h) : h(h), c(h->c), tc(h->tc()) {}

    // operand buffers for an M x K product: pre-split into the tensor-core
    // scratch when that path runs, else fp32 rows in `col`
    bool split(int M, int K) const { return linear_takes_split(c.dtype, M, K, tc); }
    bf16* hi() const { return (bf16*)tc.base; }
    bf16* lo(int M, int K) const { return (bf16*)tc.base + (size_t)M * K; }

    int gather(const float* x, int M, int Cin, int K, int d, int rev, const float2* ab, float** X) {
        const size_t n = (size_t)M * K * (Cin / 4);
        if (split(M, K * Cin)) {
            launch_pdl(gather_kernel, grid_for(n, 256), 256, 0, h->st, x, M, Cin, K, d, rev, ab, nullptr, hi(),
                                                               lo(M, K * Cin));
            *X = nullptr;
        } else {
            float* col = h->p<float>(h->col);
            launch_pdl(gather_kernel, grid_for(n, 256), 256, 0, h->st, x, M, Cin, K, d, rev, ab, col, nullptr, nullptr);
            *X = col;
        }
        ++launches;
        CC(cudaGetLastError());
        return Q3_OK;
    }
    int linear(const void* W, int N, int K, const float* X, int M, float* Y, const float* bias, int acc) {
        CC(launch_linear(c.dtype, W, N, K, X, K, M, Y, N, bias, acc, tc, h->errp(), h->st));
        launches += (X && split(M, K)) ? 2 : 1;
        return Q3_OK;
    }

    int run(const int32_t* codes_dev, int T, float* wav) {
        const int D = c.hidden, F = c.ffn, Dc = c.codebook_dim, L = c.n_layers, NQ = c.n_codebooks;
        const size_t e = esz(c.dtype);
        float* zs = h->p<float>(h->zs);
        float* za = h->p<float>(h->za);
        float* x = h->p<float>(h->x);
        float* qkv = h->p<float>(h->qkv);
        float* att = h->p<float>(h->att);
        float* tmp = h->p<float>(h->tmp);
        float* op = h->p<float>(h->op);
        float* act = h->p<float>(h->act);
        const q3codec_weights& w = h->w;
        // SplitRVQ dequantisation and the two output projections
        if (c.dtype == Q3_BF16)
            launch_pdl(dequant_kernel<bf16>, T, 256, 0, h->st, codes_dev, NQ, c.codebook_size, Dc, (const bf16*)w.codebooks,
                                                       zs, za, h->errp());
        else
            launch_pdl(dequant_kernel<float>, T, 256, 0, h->st, codes_dev, NQ, c.codebook_size, Dc, (const float*)w.codebooks,
                                                        zs, za, h->errp());
        ++launches;
        CC(cudaGetLastError());
        int r;
        if ((r = linear(w.proj_sem, D, Dc, zs, T, x, nullptr, 0))) return r;
        if ((r = linear(w.proj_ac, D, Dc, za, T, x, nullptr, 1))) return r;
        // transformer
        for (int l = 0; l < L; ++l) {
            const char* wqkv = (const char*)w.wqkv + (size_t)l * 3 * D * D * e;
            const char* wo = (const char*)w.wo + (size_t)l * D * D * e;
            const char* wgu = (const char*)w.wgu + (size_t)l * 2 * F * D * e;
            const char* wd = (const char*)w.wd + (size_t)l * D * F * e;
            if ((r = norm(x, T, (const float*)w.attn_norm + (size_t)l * D, op))) return r;
            if ((r = linear(wqkv, 3 * D, D, split(T, D) ? nullptr : op, T, qkv, nullptr, 0))) return r;
            launch_pdl(rope64_kernel, T, 256, 0, h->st, qkv, D, c.rope_theta);
            launch_pdl(window_attn_kernel, dim3(T, c.n_heads), 128, std::min(T, c.window) * sizeof(float), h->st, 
                qkv, D, c.window, att);
            launches += 2;
            CC(cudaGetLastError());
            if ((r = linear(wo, D, D, att, T, tmp, nullptr, 0))) return r;
            if ((r = scale_add(x, tmp, (const float*)w.ls_attn + (size_t)l * D, (size_t)T * D, D))) return r;
            if ((r = norm(x, T, (const float*)w.mlp_norm + (size_t)l * D, op))) return r;
            CC(launch_linear_gated(c.dtype, wgu, F, D, split(T, D) ? nullptr : op, D, T, act, F, tc, h->errp(),
                                   h->st));
            ++launches;
            if ((r = linear(wd, D, F, act, T, tmp, nullptr, 0))) return r;
            if ((r = scale_add(x, tmp, (const float*)w.ls_mlp + (size_t)l * D, (size_t)T * D, D))) return r;
        }
        float* A = h->p<float>(h->bufA);
        float* B = h->p<float>(h->bufB);
        CC(launch_rmsnorm(x, D, T, (const float*)w.final_norm, D, c.rms_eps, A, D, nullptr, 0, nullptr, h->st));
        ++launches;
        // upsampling: transposed conv (kernel = stride = 2) + ConvNeXt
        int n = T;
        for (int u = 0; u < c.n_up; ++u) {
            const char* uw = (const char*)w.up_w + (size_t)u * 2 * D * D * e;
            if ((r = linear(uw, 2 * D, D, A, n, B, h->p<float>(h->rep) + h->rep_up[u], 0))) return r;
            n *= 2;
            std::swap(A, B);   // A = x [n][D]
            const int F2 = c.up_ffn;
            const bool sp = split(n, D);
            float* nrm = h->p<float>(h->col);
            launch_pdl(dwconv_ln_kernel, n, 256, D * sizeof(float), h->st, 
                A, D, (const float*)w.dw_w + (size_t)u * D * 7, (const float*)w.dw_b + (size_t)u * D,
                (const float*)w.ln_w + (size_t)u * D, (const float*)w.ln_b + (size_t)u * D, c.ln_eps,
                sp ? nullptr : nrm, sp ? hi() : nullptr, sp ? lo(n, D) : nullptr);
            ++launches;
            CC(cudaGetLastError());
            if ((r = linear((const char*)w.fc1_w + (size_t)u * F2 * D * e, F2, D, sp ? nullptr : nrm, n, B,
                            (const float*)w.fc1_b + (size_t)u * F2, 0))) return r;
            const bool sp2 = split(n, F2);
            launch_pdl(gelu_kernel, grid_for((size_t)n * F2, 256), 256, 0, h->st, B, (size_t)n * F2, B, sp2 ? hi() : nullptr,
                                                                          sp2 ? lo(n, F2) : nullptr);
            ++launches;
            CC(cudaGetLastError());
            float* y = h->p<float>(h->col);
            if ((r = linear((const char*)w.fc2_w + (size_t)u * D * F2 * e, D, F2, sp2 ? nullptr : B, n, y,
                            (const float*)w.fc2_b + (size_t)u * D, 0))) return r;
            if ((r = scale_add(A, y, (const float*)w.gamma + (size_t)u * D, (size_t)n * D, D))) return r;
        }
        // vocoder input convolution
        int C = c.dac_channels;
        float* X;
        if ((r = gather(A, n, D, 7, 1, 0, nullptr, &X))) return r;
        if ((r = linear(w.in_w, C, 7 * D, X, n, B, (const float*)w.in_b, 0))) return r;
        std::swap(A, B);
        float* R = h->p<float>(h->bufR);
        const float2* snk = h->p<float2>(h->snk);
        static const int dil[3] = {1, 3, 9};
        for (int b = 0; b < c.n_blocks; ++b) {
            const int s = c.strides[b], Co = C / 2;
            if ((r = gather(A, n, C, 2, 1, 1, snk + h->snk_blk[b], &X))) return r;
            if ((r = linear(w.blk[b][2], s * Co, 2 * C, X, n, B, h->p<float>(h->rep) + h->rep_blk[b], 0))) return r;
            n *= s;
            C = Co;
            std::swap(A, B);
            for (int u = 0; u < 3; ++u) {
                const void* const* p = w.unit[b][u];
                if ((r = gather(A, n, C, 7, dil[u], 0, snk + h->snk_unit[b][u][0], &X))) return r;
                if ((r = linear(p[2], C, 7 * C, X, n, R, (const float*)p[3], 0))) return r;
                if ((r = gather(R, n, C, 1, 1, 0, snk + h->snk_unit[b][u][1], &X))) return r;
                if ((r = linear(p[6], C, C, X, n, A, (const float*)p[7], 1))) return r;
            }
        }
        const int warps = 8;
        if (c.dtype == Q3_BF16)
            launch_pdl(out_conv_kernel<bf16>, (n + warps - 1) / warps, 32 * warps, 0, h->st, 
                A, n, C, snk + h->snk_out, (const bf16*)w.out_w, (const float*)w.out_bias, wav);
        else
            launch_pdl(out_conv_kernel<float>, (n + warps - 1) / warps, 32 * warps, 0, h->st, 
                A, n, C, snk + h->snk_out, (const float*)w.out_w, (const float*)w.out_bias, wav);
        ++launches;
        CC(cudaGetLastError());
        return Q3_OK;
    }

    int launches = 0;

private:
    int norm(const float* x, int T, const float* wn, float* op) {
        const int D = c.hidden;
        if (split(T, D)) CC(launch_rmsnorm_split(x, D, T, wn, D, c.rms_eps, tc, h->st));
        else CC(launch_rmsnorm(x, D, T, wn, D, c.rms_eps, op, D, nullptr, 0, nullptr, h->st));
        ++launches;
        return Q3_OK;
    }
    int scale_add(float* x, const float* y, const float* g, size_t n, int C) {
        launch_pdl(scale_add_kernel, grid_for(n, 256), 256, 0, h->st, x, y, g, n, C);
        ++launches;
        CC(cudaGetLastError());
        return Q3_OK;
    }

    q3codec* h;
    const q3codec_config& c;
    TcScratch tc;
};

// decode codes [T][NQ] (host or device) and copy the samples of frames
// keep_from.. to wav (host or device)
int decode_window(q3codec* h, const int32_t* codes, int T, int keep_from, float* wav) {
    if (T < 1 || T > h->c.max_frames) return cfail(h, Q3_ERR_ARG, "T = %d outside 1..max_frames (%d)", T, h->c.max_frames);
    if (keep_from < 0 || keep_from > T) return cfail(h, Q3_ERR_ARG, "keep_from = %d outside 0..T", keep_from);
    if (!codes || (!wav && keep_from < T)) return cfail(h, Q3_ERR_ARG, "NULL codes or wav");
    const int NQ = h->c.n_codebooks;
    int32_t* cd = h->p<int32_t>(h->codes);
    if (is_dev(codes)) {
        CC(cudaMemcpyAsync(cd, codes, (size_t)T * NQ * 4, cudaMemcpyDeviceToDevice, h->st));
    } else {
        for (int i = 0; i < T * NQ; ++i)
            if (codes[i] < 0 || codes[i] >= h->c.codebook_size)
                return cfail(h, Q3_ERR_ARG, "code %d at [%d][%d] outside the codebook", codes[i], i / NQ, i % NQ);
        CC(cudaMemcpyAsync(cd, codes, (size_t)T * NQ * 4, cudaMemcpyHostToDevice, h->st));
    }
    CC(cudaMemsetAsync(h->errp(), 0, 16, h->st));
    Window win(h);
    float* wd = h->p<float>(h->wav);
    int r = win.run(cd, T, wd);
    if (r) return r;
    h->kernels = win.launches;
    const size_t n0 = (size_t)keep_from * h->spf, n = (size_t)(T - keep_from) * h->spf;
    if (n) CC(cudaMemcpyAsync(wav, wd + n0, n * 4, cudaMemcpyDefault, h->st));
    int err = 0;
    CC(cudaMemcpyAsync(&err, h->errp(), 4, cudaMemcpyDeviceToHost, h->st));
    CC(cudaStreamSynchronize(h->st));
    if (err & ERRB_BOUNDS) return cfail(h, Q3_ERR_BOUNDS, "a device code was outside the codebook");
    if (err & ERRB_TIMEOUT) return cfail(h, Q3_ERR_TIMEOUT, "a tensor-core wait gave up");
    return Q3_OK;
}

}  // namespace

extern "C" {

size_t q3codec_workspace_bytes(const q3codec_config* cfg) {
    if (!cfg_ok(cfg, nullptr)) return 0;
    q3codec h;
    h.c = *cfg;
    layout(&h);
    return h.total;
}

int q3codec_create(const q3codec_config* cfg, const q3codec_weights* w, void* workspace, size_t ws_bytes,
                   void* stream, q3codec_t** out) {
    if (!out) return Q3_ERR_ARG;
    *out = nullptr;
    std::string why;
    if (!cfg_ok(cfg, &why)) return Q3_ERR_ARG;
    if (!w || !workspace) return Q3_ERR_ARG;
    q3codec* h = new q3codec;
    h->c = *cfg;
    h->w = *w;
    layout(h);
    if (ws_bytes < h->total || ((uintptr_t)workspace % ALIGN)) { delete h; return Q3_ERR_ARG; }
    // every weight the configuration uses must be given
    const void* need[] = {w->codebooks, w->proj_sem, w->proj_ac, w->final_norm, w->in_w, w->in_b, w->out_a, w->out_b,
                          w->out_w, w->out_bias};
    for (const void* p : need)
        if (!p) { delete h; return Q3_ERR_ARG; }
    if (cfg->n_layers > 0 && (!w->attn_norm || !w->wqkv || !w->wo || !w->ls_attn || !w->mlp_norm || !w->wgu ||
                              !w->wd || !w->ls_mlp)) { delete h; return Q3_ERR_ARG; }
    if (cfg->n_up > 0 && (!w->up_w || !w->up_b || !w->dw_w || !w->dw_b || !w->ln_w || !w->ln_b || !w->fc1_w ||
                          !w->fc1_b || !w->fc2_w || !w->fc2_b || !w->gamma)) { delete h; return Q3_ERR_ARG; }
    for (int b = 0; b < cfg->n_blocks; ++b) {
        for (int i = 0; i < 4; ++i) if (!w->blk[b][i]) { delete h; return Q3_ERR_ARG; }
        for (int u = 0; u < 3; ++u)
            for (int i = 0; i < 8; ++i) if (!w->unit[b][u][i]) { delete h; return Q3_ERR_ARG; }
    }
    h->ws = (char*)workspace;
    h->st = (cudaStream_t)stream;
    // SnakeBeta tables and repeated biases
    auto fill = [&]() -> int {
        float2* snk = h->p<float2>(h->snk);
        int C = cfg->dac_channels;
        for (int b = 0; b < cfg->n_blocks; ++b) {
            const int Co = C / 2;
            snake_table_kernel<<<(C + 255) / 256, 256, 0, h->st>>>((const float*)w->blk[b][0], (const float*)w->blk[b][1],
                                                                   C, snk + h->snk_blk[b]);
            for (int u = 0; u < 3; ++u) {
                snake_table_kernel<<<(Co + 255) / 256, 256, 0, h->st>>>(
                    (const float*)w->unit[b][u][0], (const float*)w->unit[b][u][1], Co, snk + h->snk_unit[b][u][0]);
                snake_table_kernel<<<(Co + 255) / 256, 256, 0, h->st>>>(
                    (const float*)w->unit[b][u][4], (const float*)w->unit[b][u][5], Co, snk + h->snk_unit[b][u][1]);
            }
            repeat_kernel<<<(Co * cfg->strides[b] + 255) / 256, 256, 0, h->st>>>(
                (const float*)w->blk[b][3], Co, cfg->strides[b], h->p<float>(h->rep) + h->rep_blk[b]);
            C = Co;
        }
        snake_table_kernel<<<(C + 255) / 256, 256, 0, h->st>>>((const float*)w->out_a, (const float*)w->out_b, C,
                                                               snk + h->snk_out);
        for (int u = 0; u < cfg->n_up; ++u)
            repeat_kernel<<<(2 * cfg->hidden + 255) / 256, 256, 0, h->st>>>(
                (const float*)w->up_b + (size_t)u * cfg->hidden, cfg->hidden, 2, h->p<float>(h->rep) + h->rep_up[u]);
        CC(cudaGetLastError());
        CC(cudaStreamSynchronize(h->st));
        return Q3_OK;
    };
    if (fill() != Q3_OK) { delete h; return Q3_ERR_CUDA; }
    *out = h;
    return Q3_OK;
}

int q3codec_samples_per_frame(const q3codec_t* h) { return h ? h->spf : 0; }

int q3codec_decode_window(q3codec_t* h, const int32_t* codes, int T, int keep_from, float* wav) {
    if (!h) return Q3_ERR_ARG;
    return decode_window(h, codes, T, keep_from, wav);
}

int q3codec_decode(q3codec_t* h, const int32_t* codes, int T, float* wav) {
    if (!h) return Q3_ERR_ARG;
    if (T < 1 || !codes || !wav) return cfail(h, Q3_ERR_ARG, "T < 1 or NULL pointer");
    if (h->c.max_frames < std::min(T, CHUNK + CONTEXT))
        return cfail(h, Q3_ERR_ARG, "max_frames %d below the chunk window %d", h->c.max_frames, std::min(T, CHUNK + CONTEXT));
    const int NQ = h->c.n_codebooks;
    for (int c0 = 0; c0 < T; c0 += CHUNK) {
        const int s0 = std::max(0, c0 - CONTEXT), e = std::min(T, c0 + CHUNK);
        const int r = decode_window(h, codes + (size_t)s0 * NQ, e - s0, c0 - s0, wav + (size_t)c0 * h->spf);
        if (r) return r;
    }
    return Q3_OK;
}

int q3codec_stream_reset(q3codec_t* h) {
    if (!h) return Q3_ERR_ARG;
    h->s_codes.clear();
    h->s_sent = 0;
    h->s_due = S_FIRST;
    h->s_final = false;
    return Q3_OK;
}

int q3codec_stream_push(q3codec_t* h, const int32_t* codes, int n, int final, float* wav, long capacity,
                        long* n_samples) {
    if (!h) return Q3_ERR_ARG;
    if (!n_samples || n < 0 || (n > 0 && !codes)) return cfail(h, Q3_ERR_ARG, "bad stream_push arguments");
    *n_samples = 0;
    if (h->s_final) return cfail(h, Q3_ERR_STATE, "stream_push after the final push");
    if (h->c.max_frames < CHUNK + CONTEXT)
        return cfail(h, Q3_ERR_ARG, "streaming needs max_frames >= %d", CHUNK + CONTEXT);
    const int NQ = h->c.n_codebooks;
    for (long i = 0; i < (long)n * NQ; ++i)
        if (codes[i] < 0 || codes[i] >= h->c.codebook_size) return cfail(h, Q3_ERR_ARG, "code outside the codebook");
    const long spf = h->spf;
    const int have = (int)(h->s_codes.size() / NQ);
    // the decodes due while these frames arrive: after frame S_FIRST, then every
    // S_EVERY, and at the end of the request
    std::vector<int> due;
    int d = h->s_due;
    for (int k = have + 1; k <= have + n; ++k)
        if (k == d) { due.push_back(k); d += S_EVERY; }
    const int total = have + n;
    if (final && total > 0 && (due.empty() || due.back() != total)) due.push_back(total);
    // room for every sample these decodes send
    const long last = due.empty() ? h->s_sent : (long)due.back() * spf;
    if (last - h->s_sent > capacity) return cfail(h, Q3_ERR_CAPACITY, "wav holds %ld samples, %ld due", capacity, last - h->s_sent);
    h->s_codes.insert(h->s_codes.end(), codes, codes + (size_t)n * NQ);
    h->s_due = d;
    if (final) h->s_final = true;
    long written = 0;
    auto emit = [&](int s0, int e) -> int {   // decode frames [s0, e), send samples from s_sent on
        const int keep = (int)(h->s_sent / spf) - s0;
        const int r = decode_window(h, h->s_codes.data() + (size_t)s0 * NQ, e - s0, keep, wav + written);
        if (r) return r;
        written += (long)(e - s0 - keep) * spf;
        h->s_sent = (long)e * spf;
        return Q3_OK;
    };
    for (int k : due) {
        const int c0 = (k - 1) / CHUNK * CHUNK;
        while (h->s_sent < (long)c0 * spf) {   // an earlier chunk's samples are not all out: finish it
            const int pc0 = (int)(h->s_sent / spf) / CHUNK * CHUNK;
            const int r = emit(std::max(0, pc0 - CONTEXT), pc0 + CHUNK);
            if (r) return r;
        }
        const int r = emit(std::max(0, c0 - CONTEXT), k);
        if (r) return r;
    }
    *n_samples = written;
    return Q3_OK;
}

int q3codec_window_kernel_count(const q3codec_t* h) { return h ? h->kernels : 0; }

const char* q3codec_last_error(const q3codec_t* h) { return h ? h->last_error.c_str() : "NULL handle"; }

void q3codec_destroy(q3codec_t* h) { delete h; }

}  // extern "C"
