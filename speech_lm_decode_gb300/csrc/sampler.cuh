// Logits processors and the draw (device code shared by the sampler kernels
// and the persistent frame kernel), one 256-thread block per selection.
//
// Talker chain (ncnn discussion 6798 section 6; ncnn discussion 6832 section
// 3.2; Mizuoto "Qwen3-TTS" page, sections "与上游一致的做法" and "速度"):
//   sign-aware repetition penalty over the row's earlier selections ->
//   EOS logit -inf while the selection index < min_new_tokens ->
//   ids [suppress_lo, suppress_hi) except EOS to -inf ->
//   greedy argmax (lowest index on ties), or temperature -> top-k -> top-p ->
//   argmax over kept ids of w_i / E_i, w_i = exp(l_i - max), E_i ~ Exp(1).
// The predictor's draws use the same steps without penalty, min_new_tokens
// and suppression.  NaN or +inf logits fail closed.
//
// Bit-exact arithmetic (the same results as any other implementation of this
// specification): penalty and temperature are single IEEE fp32 operations;
// exp and log are this file's own fp32 restatements (Cody-Waite reduction with
// a degree-8 Taylor polynomial; atanh series), using only correctly rounded
// + - * / with no fused multiply-add; the top-p prefix sums are exact integer
// sums of floor(w_i * 2^40), so they do not depend on summation order; the
// noise is Philox4x32-10 (Salmon et al., SC'11) keyed by the row seed with
// counter (token, step, frame, row), u = (2*(x0 >> 9) + 1) * 2^-24.
#pragma once
#include "common.cuh"

namespace q3 {


// ------------------------------------------------------------------ noise
__device__ __forceinline__ uint32_t philox_x0(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                              uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c0;
}

__device__ __forceinline__ float noise_uniform(uint64_t seed, uint32_t row, uint32_t frame, uint32_t step,
                                               uint32_t token) {
    const uint32_t x0 = philox_x0(token, step, frame, row, (uint32_t)seed, (uint32_t)(seed >> 32));
    return __fmul_rn((float)(2u * (x0 >> 9) + 1u), 1.0f / 16777216.0f);
}

// ------------------------------------------------------------------ exp / log
constexpr float kLn2Hi = 0.693145751953125f;          // ln2 split: 16 leading bits
constexpr float kLn2Lo = 1.428606765330187e-06f;       // ln2 - kLn2Hi
constexpr float kInvLn2 = 1.44269502162933349609375f;  // 1/ln2 rounded to fp32

__device__ __forceinline__ float spec_expf(float x) {  // x <= 0
    if (x < -86.0f) return 0.0f;
    const float n = rintf(__fmul_rn(x, kInvLn2));
    const float r = __fsub_rn(__fsub_rn(x, __fmul_rn(n, kLn2Hi)), __fmul_rn(n, kLn2Lo));
    float p = 1.0f / 40320.0f;
    p = __fadd_rn(1.0f / 5040.0f, __fmul_rn(r, p));
    p = __fadd_rn(1.0f / 720.0f, __fmul_rn(r, p));
    p = __fadd_rn(1.0f / 120.0f, __fmul_rn(r, p));
    p = __fadd_rn(1.0f / 24.0f, __fmul_rn(r, p));
    p = __fadd_rn(1.0f / 6.0f, __fmul_rn(r, p));
    p = __fadd_rn(0.5f, __fmul_rn(r, p));
    p = __fadd_rn(1.0f, __fmul_rn(r, p));
    p = __fadd_rn(1.0f, __fmul_rn(r, p));
    const int ni = (int)n;
    return __fmul_rn(p, __uint_as_float((uint32_t)(ni + 127) << 23));
}

__device__ __forceinline__ float spec_logf(float u) {  // u in (0, 1), normal
    const uint32_t bits = __float_as_uint(u);
    int e = (int)((bits >> 23) & 0xFF) - 126;
    float f = __uint_as_float((bits & 0x007FFFFFu) | 0x3F000000u);
    if (f < 0.70710678f) { f = __fmul_rn(f, 2.0f); e -= 1; }
    const float t = __fdiv_rn(__fsub_rn(f, 1.0f), __fadd_rn(f, 1.0f));
    const float s = __fmul_rn(t, t);
    float p = 2.0f / 9.0f;
    p = __fadd_rn(2.0f / 7.0f, __fmul_rn(s, p));
    p = __fadd_rn(2.0f / 5.0f, __fmul_rn(s, p));
    p = __fadd_rn(2.0f / 3.0f, __fmul_rn(s, p));
    p = __fadd_rn(2.0f, __fmul_rn(s, p));
    const float lf = __fmul_rn(t, p);
    const float ef = (float)e;
    return __fadd_rn(__fadd_rn(__fmul_rn(ef, kLn2Lo), lf), __fmul_rn(ef, kLn2Hi));
}

// ------------------------------------------------------------------ block helpers (256 threads)
// The draw runs on threads 0..255 of the block and synchronises them with
// named barrier 1, so a kernel may keep other warps (e.g. a copy producer)
// outside it.
constexpr int ST = 256;

__device__ __forceinline__ void samp_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ int samp_sync_or(int v) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.or.pred q, 1, 256, p;\n\t"
        "selp.s32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v)
        : "memory");
    return r;
}

// Scratch of one draw over at most VMAX logits.
template <int VMAX>
struct SampSmemT {
    float l[VMAX];
    unsigned long long key[VMAX];
    int kept[VMAX];
    unsigned char keep_flag[VMAX];
    int hist[256];
    long long scan[ST];
    float red_f[ST / 32];
    int red_i[ST / 32];
    int n_kept, sel_bin, sel_above, result;
    float mx;
    long long Z;
};
using SampSmem = SampSmemT<MAX_VOCAB>;



__device__ __forceinline__ bool better(float a, int ia, float b, int ib) { return a > b || (a == b && ia < ib); }

// Argmax over (value desc, index asc); the result index is returned to all threads.
template <class S>
__device__ __forceinline__ int block_argmax(S& sm, float v, int i) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
        if (better(v2, i2, v, i)) { v = v2; i = i2; }
    }
    const int warp = threadIdx.x >> 5;
    samp_sync();
    if ((threadIdx.x & 31) == 0) { sm.red_f[warp] = v; sm.red_i[warp] = i; }
    samp_sync();
    if (threadIdx.x == 0) {
        float bv = sm.red_f[0];
        int bi = sm.red_i[0];
        for (int w = 1; w < ST / 32; ++w)
            if (better(sm.red_f[w], sm.red_i[w], bv, bi)) { bv = sm.red_f[w]; bi = sm.red_i[w]; }
        sm.result = bi;
    }
    samp_sync();
    return sm.result;
}

template <class S>
__device__ __forceinline__ float block_max(S& sm, float v) {
    v = warp_max(v);
    samp_sync();
    if ((threadIdx.x & 31) == 0) sm.red_f[threadIdx.x >> 5] = v;
    samp_sync();
    float r = sm.red_f[0];
    for (int w = 1; w < ST / 32; ++w) r = fmaxf(r, sm.red_f[w]);
    samp_sync();
    return r;
}

// Inclusive scan of one int64 per thread (thread order); also returns the total.
template <class S>
__device__ __forceinline__ long long block_scan_ll(S& sm, long long v, long long* total) {
    sm.scan[threadIdx.x] = v;
    samp_sync();
    for (int o = 1; o < ST; o <<= 1) {
        const long long add = threadIdx.x >= o ? sm.scan[threadIdx.x - o] : 0;
        samp_sync();
        sm.scan[threadIdx.x] += add;
        samp_sync();
    }
    const long long r = sm.scan[threadIdx.x];
    *total = sm.scan[ST - 1];
    samp_sync();
    return r;
}

__device__ __forceinline__ uint32_t order_key(float f) {  // larger float -> larger key
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float order_key_inv(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// k-th largest of l[0..V) counting multiplicity (1 <= k <= V): MSB-first radix
// select over the order-preserving 32-bit keys, 8 bits per pass.
template <class S>
__device__ __forceinline__ float kth_largest(S& sm, int V, int k) {
    uint32_t prefix = 0, pmask = 0;
    int kk = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        sm.hist[threadIdx.x] = 0;
        samp_sync();
        for (int i = threadIdx.x; i < V; i += ST) {
            const uint32_t key = order_key(sm.l[i]);
            if ((key & pmask) == prefix) atomicAdd(&sm.hist[(key >> shift) & 255u], 1);
        }
        samp_sync();
        // thread t owns bin 255 - t: inclusive scan gives counts from the top
        const int c = sm.hist[255 - threadIdx.x];
        long long tot;
        const long long incl = block_scan_ll(sm, c, &tot);
        if (incl - c < kk && kk <= incl) { sm.sel_bin = 255 - threadIdx.x; sm.sel_above = (int)(incl - c); }
        samp_sync();
        prefix |= (uint32_t)sm.sel_bin << shift;
        pmask |= 255u << shift;
        kk -= sm.sel_above;
        samp_sync();
    }
    return order_key_inv(prefix);
}

struct DrawCfg {
    int do_sample;
    float temperature;
    int top_k;
    float top_p;
};

// One selection.  All 256 threads call it; returns the id (or -1 when the
// logits hold NaN / +inf or no finite value) to every thread.
//   lg: the raw logits in global memory, or nullptr when sm.l[0, V) holds them
//       (each thread i of the block must have written the entries i, i + 256, ...).
//   seen_bits / seen_bytes: ids drawn before (penalty); one of them or neither.
//   S: a SampSmemT<VMAX> with V <= VMAX.
template <class S>
static __device__ __noinline__ int sample_row(S& sm, const float* __restrict__ lg, int V, DrawCfg d, bool talker, float penalty,
                          const uint32_t* seen_bits, const uint8_t* seen_bytes, int sel, int min_new, int eos,
                          int sup_lo, int sup_hi, uint64_t seed, uint32_t row, uint32_t frame, uint32_t step) {
    const int tid = threadIdx.x;
    int bad = 0;
    for (int i = tid; i < V; i += ST) {
        // logits may come from other CTAs of the same launch (read at L2); with
        // lg == nullptr the caller has already placed them in sm.l
        float v = lg ? __ldcg(lg + i) : sm.l[i];
        bad |= (isnan(v) || v == INFINITY) ? 1 : 0;
        if (talker) {
            const bool seen = seen_bits ? ((seen_bits[i >> 5] >> (i & 31)) & 1u) : (seen_bytes ? seen_bytes[i] : 0);
            if (seen && penalty != 1.0f) v = v < 0.0f ? __fmul_rn(v, penalty) : __fdiv_rn(v, penalty);
            if (sel < min_new && i == eos) v = -INFINITY;
            if (i >= sup_lo && i < sup_hi && i != eos) v = -INFINITY;
        }
        sm.l[i] = v;
    }
    if (samp_sync_or(bad)) return -1;

    if (!d.do_sample) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int i = tid; i < V; i += ST)
            if (better(sm.l[i], i, bv, bi)) { bv = sm.l[i]; bi = i; }
        return block_argmax(sm, bv, bi);
    }

    if (d.temperature != 1.0f)
        for (int i = tid; i < V; i += ST) sm.l[i] = __fdiv_rn(sm.l[i], d.temperature);
    samp_sync();

    float thr = -INFINITY;
    if (d.top_k > 0 && d.top_k < V) thr = kth_largest(sm, V, d.top_k);

    if (tid == 0) sm.n_kept = 0;
    samp_sync();
    float lmax = -INFINITY;
    for (int i = tid; i < V; i += ST) {
        const float v = sm.l[i];
        if (v != -INFINITY && v >= thr) {
            sm.kept[atomicAdd(&sm.n_kept, 1)] = i;
            lmax = fmaxf(lmax, v);
        }
    }
    samp_sync();
    const int nk = sm.n_kept;
    if (nk == 0) return -1;
    const float mx = block_max(sm, lmax);
    for (int j = tid; j < nk; j += ST) sm.keep_flag[j] = 1;
    samp_sync();

    if (d.top_p < 1.0f) {
        // order kept ids by (l desc, id asc): ascending sort of composite keys
        int npad = 1;
        while (npad < nk) npad <<= 1;
        for (int j = tid; j < npad; j += ST) {
            if (j < nk) {
                const int i = sm.kept[j];
                float v = sm.l[i];
                if (v == 0.0f) v = 0.0f;  // -0 and +0 order as equal
                sm.key[j] = ((unsigned long long)(~order_key(v)) << 32) | (unsigned)i;
            } else {
                sm.key[j] = ~0ull;
            }
        }
        samp_sync();
        for (int size = 2; size <= npad; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int t = tid; t < npad / 2; t += ST) {
                    const int lo = (t / stride) * 2 * stride + (t % stride);
                    const int hi = lo + stride;
                    const bool asc = (lo & size) == 0;
                    const unsigned long long a = sm.key[lo], b = sm.key[hi];
                    if ((a > b) == asc) { sm.key[lo] = b; sm.key[hi] = a; }
                }
                samp_sync();
            }
        }
        // exact integer prefix sums of W = floor(w * 2^40) in sorted order
        const int per = (nk + ST - 1) / ST;
        const int s0 = min(tid * per, nk), s1 = min(s0 + per, nk);
        long long local = 0;
        for (int j = s0; j < s1; ++j) {
            const int i = (int)(sm.key[j] & 0xffffffffu);
            local += (long long)floor(__dmul_rn((double)spec_expf(__fsub_rn(sm.l[i], mx)), 1099511627776.0));
        }
        long long Z;
        long long c = block_scan_ll(sm, local, &Z) - local;
        const double limit = __dmul_rn((double)d.top_p, (double)Z);
        for (int j = s0; j < s1; ++j) {
            const int i = (int)(sm.key[j] & 0xffffffffu);
            sm.kept[j] = i;
            sm.keep_flag[j] = (j == 0 || (double)c < limit) ? 1 : 0;
            c += (long long)floor(__dmul_rn((double)spec_expf(__fsub_rn(sm.l[i], mx)), 1099511627776.0));
        }
        samp_sync();
    }

    float bs = -INFINITY;
    int bi = 0x7fffffff;
    for (int j = tid; j < nk; j += ST) {
        if (!sm.keep_flag[j]) continue;
        const int i = sm.kept[j];
        const float u = noise_uniform(seed, row, frame, step, (uint32_t)i);
        const float E = -spec_logf(u);
        const float s = __fdiv_rn(spec_expf(__fsub_rn(sm.l[i], mx)), E);
        if (better(s, i, bs, bi)) { bs = s; bi = i; }
    }
    return block_argmax(sm, bs, bi);
}

}  // namespace q3
