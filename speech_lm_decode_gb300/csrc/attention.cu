// QK-norm + RoPE + KV append, and split-KV grouped-query decode attention
// over the static per-row cache [maxB][nkv][cap][128].
//
// The method: per-head RMSNorm of q and of k, each with its own weight
// (q and k normalised separately, Mizuoto "Qwen3-TTS" page, section "速度"),
// rotate-half RoPE at the absolute position with inv_freq held in fp32
// (same page, section "对照结果"), GQA where q head h reads kv head
// h / (nq/nkv) (repeat_interleave over heads, ncnn discussion 6798,
// section 2), causal softmax over positions 0..pos.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "pdl.cuh"

namespace q3 {

// ------------------------------------------------------------------ QK-norm, RoPE, KV append
// grid: M tokens; block: 32 * (nq + nkv) threads.  Warp w < nq: q head w;
// otherwise k head w - nq (and the matching v head is copied to the cache).
// Lane l holds head elements l, l+32, l+64, l+96: the RoPE pairs (j, j+64)
// for j = l and j = l+32 stay inside the lane.
template <typename T>
__global__ void qk_rope_kv_kernel(float* __restrict__ qkv, int ldq, int nq, int nkv, const float* __restrict__ qn,
                                  const float* __restrict__ kn, float eps, const float2* __restrict__ rope,
                                  int rope_rows, T* __restrict__ Kc, T* __restrict__ Vc, int cap,
                                  const int* __restrict__ tok_row, const int* __restrict__ tok_pos, int* err) {
    pdl_wait();
    pdl_trigger();
    const int m = blockIdx.x;
    const int pos = tok_pos[m];
    if (pos < 0) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (pos >= cap || pos >= rope_rows) {
        if (threadIdx.x == 0) atomicOr(err, ERRB_BOUNDS);
        return;
    }
    const int row = tok_row[m];
    float* t = qkv + (size_t)m * ldq;
    const bool is_q = warp < nq;
    const int head = is_q ? warp : warp - nq;
    float* src = t + (size_t)(is_q ? head : nq + head) * HD;
    const float* wn = is_q ? qn : kn;
    float e[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) e[i] = src[lane + 32 * i];
    float ss = warp_sum(e[0] * e[0] + e[1] * e[1] + e[2] * e[2] + e[3] * e[3]);
    const float r = 1.0f / sqrtf(ss / (float)HD + eps);
#pragma unroll
    for (int i = 0; i < 4; ++i) e[i] = e[i] * r * wn[lane + 32 * i];
    const float2 cs0 = rope[(size_t)pos * (HD / 2) + lane];
    const float2 cs1 = rope[(size_t)pos * (HD / 2) + lane + 32];
    float a = e[0], b = e[2];
    e[0] = a * cs0.x - b * cs0.y;
    e[2] = b * cs0.x + a * cs0.y;
    a = e[1]; b = e[3];
    e[1] = a * cs1.x - b * cs1.y;
    e[3] = b * cs1.x + a * cs1.y;
    if (is_q) {
#pragma unroll
        for (int i = 0; i < 4; ++i) src[lane + 32 * i] = e[i];
    } else {
        const size_t off = (((size_t)row * nkv + head) * cap + pos) * HD;
        const float* v = t + (size_t)(nq + nkv + head) * HD;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            Kc[off + lane + 32 * i] = from_f<T>(e[i]);
            Vc[off + lane + 32 * i] = from_f<T>(v[lane + 32 * i]);
        }
    }
}

cudaError_t launch_qk_rope_kv(int dtype, float* qkv, int ldq, int M, int nq, int nkv, const float* q_norm,
                              const float* k_norm, float eps, const float* rope_cs, int rope_rows, void* Kc, void* Vc,
                              int cap, const int* tok_row, const int* tok_pos, int* err, cudaStream_t st) {
    if (M <= 0) return cudaSuccess;
    const int threads = 32 * (nq + nkv);
    if (dtype == Q3_BF16)
        launch_pdl(qk_rope_kv_kernel<bf16>, M, threads, 0, st, qkv, ldq, nq, nkv, q_norm, k_norm, eps, (const float2*)rope_cs,
                                                       rope_rows, (bf16*)Kc, (bf16*)Vc, cap, tok_row, tok_pos, err);
    else
        launch_pdl(qk_rope_kv_kernel<float>, M, threads, 0, st, qkv, ldq, nq, nkv, q_norm, k_norm, eps,
                                                        (const float2*)rope_cs, rope_rows, (float*)Kc, (float*)Vc, cap,
                                                        tok_row, tok_pos, err);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ split-KV attention
// grid (n_splits, nkv, M), 128 threads.  8 lanes cover one cached position
// (16 dims each), a warp walks 4 positions at a time, the block 16.  Each
// 8-lane group keeps an online softmax (running max, sum, weighted V) per q
// head of the kv group; groups then warps are merged, and the block writes
// its unnormalised partial for the split.
template <typename T, int GQ>
__global__ void __launch_bounds__(128) attn_split_kernel(const float* __restrict__ qkv, int ldq, int nq, int nkv,
                                                         const T* __restrict__ Kc, const T* __restrict__ Vc, int cap,
                                                         const int* __restrict__ tok_row,
                                                         const int* __restrict__ tok_pos, int n_splits,
                                                         float* __restrict__ pm, float* __restrict__ pl,
                                                         float* __restrict__ pacc) {
    pdl_wait();
    pdl_trigger();
    const int split = blockIdx.x, g = blockIdx.y, m = blockIdx.z;
    const int pos = tok_pos[m];
    if (pos < 0) return;
    const int n = pos + 1;
    const int chunk = (n + n_splits - 1) / n_splits;
    const int j0 = split * chunk, j1 = min(n, j0 + chunk);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane & 7, grp = lane >> 3;
    const int d0 = sub * 16;
    const float scale = 0.08838834764831845f;  // 1/sqrt(128)

    float q[GQ][16];
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
        const float* qs = qkv + (size_t)m * ldq + (size_t)(g * GQ + hh) * HD + d0;
#pragma unroll
        for (int i = 0; i < 16; ++i) q[hh][i] = qs[i] * scale;
    }
    float mx[GQ], l[GQ], acc[GQ][16];
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
        mx[hh] = -INFINITY; l[hh] = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[hh][i] = 0.f;
    }
    const size_t base = ((size_t)tok_row[m] * nkv + g) * cap * HD;
    // the trip count is uniform over the warp (every lane runs the shuffles);
    // a group whose position is past the split's end only skips the update
    for (int jb = j0 + warp * 4; jb < j1; jb += 16) {
        const int j = jb + grp;
        const bool valid = j < j1;
        float k[16], v[16];
        if (valid) {
            float a[8], b[8];
            load8(Kc + base + (size_t)j * HD + d0, a);
            load8(Kc + base + (size_t)j * HD + d0 + 8, b);
#pragma unroll
            for (int i = 0; i < 8; ++i) { k[i] = a[i]; k[8 + i] = b[i]; }
            load8(Vc + base + (size_t)j * HD + d0, a);
            load8(Vc + base + (size_t)j * HD + d0 + 8, b);
#pragma unroll
            for (int i = 0; i < 8; ++i) { v[i] = a[i]; v[8 + i] = b[i]; }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) { k[i] = 0.f; v[i] = 0.f; }
        }
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) s = fmaf(q[hh][i], k[i], s);
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            s += __shfl_xor_sync(0xffffffffu, s, 4);
            if (valid) {
                const float mn = fmaxf(mx[hh], s);
                const float c = expf(mx[hh] - mn);
                const float p = expf(s - mn);
                l[hh] = l[hh] * c + p;
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[hh][i] = fmaf(p, v[i], acc[hh][i] * c);
                mx[hh] = mn;
            }
        }
    }
    // merge the 4 position groups of the warp (lanes sub, sub+8, sub+16, sub+24)
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
        float ma = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 8));
        ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 16));
        const float c = (ma == -INFINITY) ? 0.f : expf(mx[hh] - ma);
        float lv = l[hh] * c;
        lv += __shfl_xor_sync(0xffffffffu, lv, 8);
        lv += __shfl_xor_sync(0xffffffffu, lv, 16);
        l[hh] = lv;
        mx[hh] = ma;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float a = acc[hh][i] * c;
            a += __shfl_xor_sync(0xffffffffu, a, 8);
            a += __shfl_xor_sync(0xffffffffu, a, 16);
            acc[hh][i] = a;
        }
    }
    __shared__ float s_m[4][GQ], s_l[4][GQ], s_acc[4][GQ][HD];
    if (grp == 0) {
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
#pragma unroll
            for (int i = 0; i < 16; ++i) s_acc[warp][hh][d0 + i] = acc[hh][i];
            if (sub == 0) { s_m[warp][hh] = mx[hh]; s_l[warp][hh] = l[hh]; }
        }
    }
    __syncthreads();
    const int t = threadIdx.x;  // one head dimension per thread
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
        float ma = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) ma = fmaxf(ma, s_m[w][hh]);
        float lsum = 0.f, a = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float c = (ma == -INFINITY) ? 0.f : expf(s_m[w][hh] - ma);
            lsum += s_l[w][hh] * c;
            a += s_acc[w][hh][t] * c;
        }
        const size_t pi = ((size_t)m * n_splits + split) * nq + g * GQ + hh;
        pacc[pi * HD + t] = a;
        if (t == 0) { pm[pi] = ma; pl[pi] = lsum; }
    }
}

// grid (M, nq), 128 threads (one head dimension each): merge the splits of
// one head into the O-projection input; skipped tokens get zeros.
__global__ void __launch_bounds__(128) attn_combine_kernel(const float* __restrict__ pm, const float* __restrict__ pl,
                                                           const float* __restrict__ pacc, int n_splits, int nq,
                                                           const int* __restrict__ tok_pos, float* __restrict__ out,
                                                           int ldo, bf16* __restrict__ hi, bf16* __restrict__ lo) {
    pdl_wait();
    pdl_trigger();
    const int m = blockIdx.x, h = blockIdx.y, t = threadIdx.x;
    float res = 0.f;
    if (tok_pos[m] >= 0) {
        float ma = -INFINITY;
        for (int s = 0; s < n_splits; ++s) ma = fmaxf(ma, pm[((size_t)m * n_splits + s) * nq + h]);
        float den = 0.f, num = 0.f;
        for (int s = 0; s < n_splits; ++s) {
            const size_t pi = ((size_t)m * n_splits + s) * nq + h;
            const float c = (pm[pi] == -INFINITY) ? 0.f : expf(pm[pi] - ma);
            den += pl[pi] * c;
            num += pacc[pi * HD + t] * c;
        }
        res = num / den;
    }
    const size_t i = (size_t)h * HD + t;
    if (hi) {
        // the O projection's tensor-core operand: bf16 high and low parts, [M][nq * 128]
        const bf16 hv = __float2bfloat16_rn(res);
        hi[(size_t)m * nq * HD + i] = hv;
        lo[(size_t)m * nq * HD + i] = __float2bfloat16_rn(res - __bfloat162float(hv));
    } else {
        out[(size_t)m * ldo + i] = res;
    }
}

// ------------------------------------------------------------------ bulk-staged decode attention (bf16 cache)
// grid (n_splits, nkv, M), 256 threads, two CTAs per SM.  A split's cached
// positions of one (row, kv head) are contiguous in the cache, so K and V
// blocks of ab::P positions are each ONE cp.async.bulk into a ring of ab::NS
// shared-memory stages (completion on an mbarrier), issued by thread 0 as far
// ahead as the ring allows: up to 96 KB of the cache in flight per CTA.
// Eight lanes cover one position: lane s holds dims 8s..8s+7 and 64+8s..64+8s+7
// (each load of the group is 128 contiguous bytes of a row, no bank
// conflict); the 32 groups take positions grp and grp + 32 of every stage and
// keep an online softmax (max, sum, weighted V) per q head of the kv group in
// fp32, rescaled once per stage.  Groups then warps are merged in a fixed
// order.  One split: the normalised output (fp32, or the O projection's bf16
// high / low operand) is written directly; more: unnormalised partials for
// attn_combine_kernel.  A wait that runs out sets the TIMEOUT bit and the CTA
// leaves after a bounded wait for its own copies.
namespace ab {
constexpr int P = 64;                 // positions per stage
constexpr int NS = 3;                 // ring stages
constexpr int NT = 256;
constexpr int NG = NT / 8;            // lane groups (one position each)
constexpr int NW = NT / 32;
constexpr size_t RING = (size_t)2 * NS * P * HD * sizeof(bf16);
constexpr size_t SMEM = RING + NS * sizeof(uint64_t);
constexpr long long WAIT_CYCLES = 2000000000LL;
static_assert(P == 2 * NG, "two positions per group and stage");

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ bool try_wait(uint64_t* b, unsigned parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(su32(b)), "r"(parity) : "memory");
    return ok != 0;
}
// the lane's 16 elements of a 128-wide bf16 row in shared memory (dims 8s..8s+7, 64+8s..64+8s+7)
__device__ __forceinline__ void row16(const bf16* row, int sub, float (&v)[16]) {
    float a[8], b[8];
    unpack_bf16x8(*reinterpret_cast<const uint4*>(row + 8 * sub), a);
    unpack_bf16x8(*reinterpret_cast<const uint4*>(row + 64 + 8 * sub), b);
#pragma unroll
    for (int i = 0; i < 8; ++i) { v[i] = a[i]; v[8 + i] = b[i]; }
}
__device__ __forceinline__ bool wait_bounded(uint64_t* b, unsigned parity) {
    if (try_wait(b, parity)) return true;
    const long long t0 = clock64();
    while (!try_wait(b, parity))
        if (clock64() - t0 > WAIT_CYCLES) return false;
    return true;
}
}  // namespace ab

template <int GQ>
__global__ void __launch_bounds__(ab::NT, 2) attn_bulk_kernel(const float* __restrict__ qkv, int ldq, int nq, int nkv,
                                                              const bf16* __restrict__ Kc, const bf16* __restrict__ Vc,
                                                              int cap, const int* __restrict__ tok_row,
                                                              const int* __restrict__ tok_pos, int n_splits,
                                                              float* __restrict__ pm, float* __restrict__ pl,
                                                              float* __restrict__ pacc, float* __restrict__ out,
                                                              int ldo, bf16* __restrict__ hi, bf16* __restrict__ lo,
                                                              int* __restrict__ err) {
    pdl_wait();
    pdl_trigger();
    using namespace ab;
    extern __shared__ __align__(128) unsigned char ab_smem[];
    bf16* sK = reinterpret_cast<bf16*>(ab_smem);
    bf16* sV = sK + NS * P * HD;
    uint64_t* full = reinterpret_cast<uint64_t*>(ab_smem + RING);
    const int split = blockIdx.x, g = blockIdx.y, m = blockIdx.z;
    const int pos = tok_pos[m];
    if (pos < 0) {
        // a skipped token: zeros in the single-split output, nothing otherwise
        if (n_splits == 1)
            for (int i = threadIdx.x; i < GQ * HD; i += NT) {
                const size_t o = (size_t)g * GQ * HD + i;
                if (hi) { hi[(size_t)m * nq * HD + o] = __float2bfloat16_rn(0.f); lo[(size_t)m * nq * HD + o] = __float2bfloat16_rn(0.f); }
                else out[(size_t)m * ldo + o] = 0.f;
            }
        return;
    }
    if (pos >= cap) {   // the host checks capacity first; never read past the row's cache
        if (threadIdx.x == 0) atomicOr(err, ERRB_BOUNDS);
        return;
    }
    const int n = pos + 1;
    const int chunk = (n + n_splits - 1) / n_splits;
    const int j0 = min(n, split * chunk), j1 = min(n, j0 + chunk);
    const int cnt = j1 - j0;
    const int nst = (cnt + P - 1) / P;
    const size_t base = (((size_t)tok_row[m] * nkv + g) * cap + j0) * HD;
    const bf16* Kg = Kc + base;
    const bf16* Vg = Vc + base;
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(&full[i])), "r"(1) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    auto issue = [&](int t) {
        const int slot = t % NS;
        const unsigned bytes = (unsigned)min(P, cnt - t * P) * HD * (unsigned)sizeof(bf16);
        unsigned long long st;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 %0, [%1], %2;"
                     : "=l"(st) : "r"(su32(&full[slot])), "r"(2 * bytes) : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     ::"r"(su32(sK + (size_t)slot * P * HD)), "l"(Kg + (size_t)t * P * HD), "r"(bytes),
                       "r"(su32(&full[slot])) : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     ::"r"(su32(sV + (size_t)slot * P * HD)), "l"(Vg + (size_t)t * P * HD), "r"(bytes),
                       "r"(su32(&full[slot])) : "memory");
    };
    if (threadIdx.x == 0)
        for (int t = 0; t < min(NS, nst); ++t) issue(t);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane & 7, grp = threadIdx.x >> 3;
    const float scale = 0.08838834764831845f;  // 1/sqrt(128)
    float q[GQ][16], acc[GQ][16], mx[GQ], l[GQ];
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
        const float* qs = qkv + (size_t)m * ldq + (size_t)(g * GQ + hh) * HD;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            q[hh][i] = qs[8 * sub + i] * scale;
            q[hh][8 + i] = qs[64 + 8 * sub + i] * scale;
        }
        mx[hh] = -INFINITY; l[hh] = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[hh][i] = 0.f;
    }
    int issued = min(NS, nst);
    bool fail = false;
    for (int t = 0; t < nst; ++t) {
        const int slot = t % NS;
        if (!fail && !wait_bounded(&full[slot], (unsigned)(t / NS) & 1u)) fail = true;
        // the shuffles below need the whole warp
        if (!__any_sync(0xffffffffu, fail)) {
            const int c = min(P, cnt - t * P);
            const bf16* ks = sK + (size_t)slot * P * HD;
            const bf16* vs = sV + (size_t)slot * P * HD;
            float s[2][GQ];
            bool val[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int pl_ = grp + NG * r;
                val[r] = pl_ < c;
                float k[16];
                if (val[r]) {
                    row16(ks + pl_ * HD, sub, k);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) k[i] = 0.f;
                }
#pragma unroll
                for (int hh = 0; hh < GQ; ++hh) {
                    float d = 0.f;
#pragma unroll
                    for (int i = 0; i < 16; ++i) d = fmaf(q[hh][i], k[i], d);
                    d += __shfl_xor_sync(0xffffffffu, d, 1);
                    d += __shfl_xor_sync(0xffffffffu, d, 2);
                    d += __shfl_xor_sync(0xffffffffu, d, 4);
                    s[r][hh] = d;
                }
            }
            if (val[0]) {   // the group's second position exists only with its first
                float v0[16], v1[16];
                row16(vs + grp * HD, sub, v0);
                if (val[1]) {
                    row16(vs + (grp + NG) * HD, sub, v1);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v1[i] = 0.f;
                }
#pragma unroll
                for (int hh = 0; hh < GQ; ++hh) {
                    const float mn = val[1] ? fmaxf(fmaxf(mx[hh], s[0][hh]), s[1][hh]) : fmaxf(mx[hh], s[0][hh]);
                    const float cf = expf(mx[hh] - mn);
                    const float p0 = expf(s[0][hh] - mn);
                    const float p1 = val[1] ? expf(s[1][hh] - mn) : 0.f;
                    l[hh] = l[hh] * cf + p0 + p1;
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[hh][i] = fmaf(p1, v1[i], fmaf(p0, v0[i], acc[hh][i] * cf));
                    mx[hh] = mn;
                }
            }
        }
        // every thread is done with this slot: refill it
        if (__syncthreads_or(fail)) { fail = true; break; }
        if (threadIdx.x == 0 && issued < nst) issue(issued);
        issued += issued < nst ? 1 : 0;
    }
    if (fail) {
        if (threadIdx.x == 0) {
            atomicOr(err, ERRB_TIMEOUT);
            // copies in flight must land before the CTA leaves
            for (int t = max(0, issued - NS); t < issued; ++t) ab::wait_bounded(&full[t % NS], (unsigned)(t / NS) & 1u);
        }
        return;
    }
    // merge the 4 groups of the warp (lanes sub, sub+8, sub+16, sub+24)
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
        float ma = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 8));
        ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 16));
        const float cf = (ma == -INFINITY) ? 0.f : expf(mx[hh] - ma);
        float lv = l[hh] * cf;
        lv += __shfl_xor_sync(0xffffffffu, lv, 8);
        lv += __shfl_xor_sync(0xffffffffu, lv, 16);
        l[hh] = lv;
        mx[hh] = ma;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float a = acc[hh][i] * cf;
            a += __shfl_xor_sync(0xffffffffu, a, 8);
            a += __shfl_xor_sync(0xffffffffu, a, 16);
            acc[hh][i] = a;
        }
    }
    // the ring is drained (every issued stage was waited on): reuse it
    float* s_acc = reinterpret_cast<float*>(ab_smem);          // [NW][GQ][HD]
    float* s_m = s_acc + NW * GQ * HD;                            // [NW][GQ]
    float* s_l = s_m + NW * GQ;
    if (lane < 8) {
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                s_acc[(warp * GQ + hh) * HD + 8 * sub + i] = acc[hh][i];
                s_acc[(warp * GQ + hh) * HD + 64 + 8 * sub + i] = acc[hh][8 + i];
            }
            if (sub == 0) { s_m[warp * GQ + hh] = mx[hh]; s_l[warp * GQ + hh] = l[hh]; }
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < GQ * HD; idx += NT) {
        const int hh = idx / HD, d = idx - hh * HD;
        float ma = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) ma = fmaxf(ma, s_m[w * GQ + hh]);
        float lsum = 0.f, a = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float cf = (ma == -INFINITY) ? 0.f : expf(s_m[w * GQ + hh] - ma);
            lsum += s_l[w * GQ + hh] * cf;
            a += s_acc[(w * GQ + hh) * HD + d] * cf;
        }
        const size_t o = (size_t)(g * GQ + hh) * HD + d;
        if (n_splits == 1) {
            const float res = a / lsum;
            if (hi) {
                const bf16 hv = __float2bfloat16_rn(res);
                hi[(size_t)m * nq * HD + o] = hv;
                lo[(size_t)m * nq * HD + o] = __float2bfloat16_rn(res - __bfloat162float(hv));
            } else {
                out[(size_t)m * ldo + o] = res;
            }
        } else {
            const size_t pi = ((size_t)m * n_splits + split) * nq + g * GQ + hh;
            pacc[pi * HD + d] = a;
            if (d == 0) { pm[pi] = ma; pl[pi] = lsum; }
        }
    }
}

// Short caches (the code predictor's 16 positions): one warp per (token, kv
// head), lane l holding dims 4l..4l+3 of each q head; positions are walked in
// order with the online softmax kept identically in every lane.  The fixed
// cost of a bulk-staged CTA (barriers, copy latency, block merge) would
// exceed this work many times over.
template <int GQ>
__global__ void __launch_bounds__(256) attn_short_kernel(const float* __restrict__ qkv, int ldq, int M, int nq, int nkv,
                                                         const bf16* __restrict__ Kc, const bf16* __restrict__ Vc,
                                                         int cap, const int* __restrict__ tok_row,
                                                         const int* __restrict__ tok_pos, float* __restrict__ out,
                                                         int ldo, bf16* __restrict__ hi, bf16* __restrict__ lo,
                                                         int* __restrict__ err) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int item = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (item >= M * nkv) return;
    const int m = item / nkv, g = item - m * nkv;
    const int pos = tok_pos[m];
    float acc[GQ][4];
    float res[GQ][4];
    if (pos >= 0 && pos < cap) {
        const float scale = 0.08838834764831845f;  // 1/sqrt(128)
        float q[GQ][4], mx[GQ], l[GQ];
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
            const float4 qv = *reinterpret_cast<const float4*>(qkv + (size_t)m * ldq + (size_t)(g * GQ + hh) * HD + 4 * lane);
            q[hh][0] = qv.x * scale; q[hh][1] = qv.y * scale; q[hh][2] = qv.z * scale; q[hh][3] = qv.w * scale;
            mx[hh] = -INFINITY; l[hh] = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[hh][i] = 0.f;
        }
        const size_t base = ((size_t)tok_row[m] * nkv + g) * cap * HD + 4 * lane;
        // eight positions' loads in flight before their arithmetic
        constexpr int U = 8;
        for (int j0 = 0; j0 <= pos; j0 += U) {
            uint2 kr[U], vr[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (j0 + u <= pos) {
                    kr[u] = *reinterpret_cast<const uint2*>(Kc + base + (size_t)(j0 + u) * HD);
                    vr[u] = *reinterpret_cast<const uint2*>(Vc + base + (size_t)(j0 + u) * HD);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (j0 + u > pos) break;   // uniform over the warp (one token per warp)
                const float k[4] = {__uint_as_float(kr[u].x << 16), __uint_as_float(kr[u].x & 0xffff0000u),
                                    __uint_as_float(kr[u].y << 16), __uint_as_float(kr[u].y & 0xffff0000u)};
                const float v[4] = {__uint_as_float(vr[u].x << 16), __uint_as_float(vr[u].x & 0xffff0000u),
                                    __uint_as_float(vr[u].y << 16), __uint_as_float(vr[u].y & 0xffff0000u)};
#pragma unroll
                for (int hh = 0; hh < GQ; ++hh) {
                    const float sc = warp_sum(fmaf(q[hh][0], k[0], fmaf(q[hh][1], k[1], fmaf(q[hh][2], k[2], q[hh][3] * k[3]))));
                    const float mn = fmaxf(mx[hh], sc);
                    const float cf = expf(mx[hh] - mn);
                    const float p = expf(sc - mn);
                    l[hh] = l[hh] * cf + p;
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[hh][i] = fmaf(p, v[i], acc[hh][i] * cf);
                    mx[hh] = mn;
                }
            }
        }
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh)
#pragma unroll
            for (int i = 0; i < 4; ++i) res[hh][i] = acc[hh][i] / l[hh];
    } else {
        if (pos >= cap && lane == 0) atomicOr(err, ERRB_BOUNDS);
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh)
#pragma unroll
            for (int i = 0; i < 4; ++i) res[hh][i] = 0.f;
    }
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
        const size_t o = (size_t)(g * GQ + hh) * HD + 4 * lane;
        if (hi) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const bf16 hv = __float2bfloat16_rn(res[hh][i]);
                hi[(size_t)m * nq * HD + o + i] = hv;
                lo[(size_t)m * nq * HD + o + i] = __float2bfloat16_rn(res[hh][i] - __bfloat162float(hv));
            }
        } else {
            *reinterpret_cast<float4*>(out + (size_t)m * ldo + o) = make_float4(res[hh][0], res[hh][1], res[hh][2], res[hh][3]);
        }
    }
}

// Decode steps over short caches with QK-norm, RoPE and the cache append
// fused in (one token per row in the launch): one warp per (token, kv head)
// normalises and rotates the group's q heads and its k head (lane l holds
// elements l, l+32, l+64, l+96, so the RoPE pairs (j, j+64) stay in the
// lane), rounds k and v to the cache type and appends them at the token's
// position, then attends over positions 0..pos (the new position from its
// registers, which equal what it stored), eight positions' loads in flight.
template <int GQ>
__global__ void __launch_bounds__(256) attn_short_fused_kernel(
    const float* __restrict__ qkv, int ldq, int M, int nq, int nkv, const float* __restrict__ qn,
    const float* __restrict__ kn, float eps, const float2* __restrict__ rope, int rope_rows, bf16* __restrict__ Kc,
    bf16* __restrict__ Vc, int cap, const int* __restrict__ tok_row, const int* __restrict__ tok_pos,
    float* __restrict__ out, int ldo, bf16* __restrict__ hi, bf16* __restrict__ lo, int* __restrict__ err) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int item = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (item >= M * nkv) return;
    const int m = item / nkv, g = item - m * nkv;
    const int pos = tok_pos[m];
    float res[GQ][4];
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh)
#pragma unroll
        for (int i = 0; i < 4; ++i) res[hh][i] = 0.f;
    if (pos >= 0 && pos < cap && pos < rope_rows) {
        const float* t = qkv + (size_t)m * ldq;
        const float2 cs0 = rope[(size_t)pos * (HD / 2) + lane];
        const float2 cs1 = rope[(size_t)pos * (HD / 2) + lane + 32];
        // RMSNorm over the head (weight wn) then rotate-half RoPE at pos
        auto norm_rope = [&](const float* src, const float* wn, float (&e)[4]) {
#pragma unroll
            for (int i = 0; i < 4; ++i) e[i] = src[lane + 32 * i];
            const float ss = warp_sum(e[0] * e[0] + e[1] * e[1] + e[2] * e[2] + e[3] * e[3]);
            const float r = 1.0f / sqrtf(ss / (float)HD + eps);
#pragma unroll
            for (int i = 0; i < 4; ++i) e[i] = e[i] * r * wn[lane + 32 * i];
            float a = e[0], b = e[2];
            e[0] = a * cs0.x - b * cs0.y;
            e[2] = b * cs0.x + a * cs0.y;
            a = e[1]; b = e[3];
            e[1] = a * cs1.x - b * cs1.y;
            e[3] = b * cs1.x + a * cs1.y;
        };
        const float scale = 0.08838834764831845f;  // 1/sqrt(128)
        float q[GQ][4];
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
            norm_rope(t + (size_t)(g * GQ + hh) * HD, qn, q[hh]);
#pragma unroll
            for (int i = 0; i < 4; ++i) q[hh][i] *= scale;
        }
        float kn4[4], kcur[4], vcur[4];
        norm_rope(t + (size_t)(nq + g) * HD, kn, kn4);
        const float* vs = t + (size_t)(nq + nkv + g) * HD;
        const size_t base = ((size_t)tok_row[m] * nkv + g) * cap * HD;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const bf16 kb = __float2bfloat16_rn(kn4[i]), vb = __float2bfloat16_rn(vs[lane + 32 * i]);
            Kc[base + (size_t)pos * HD + lane + 32 * i] = kb;
            Vc[base + (size_t)pos * HD + lane + 32 * i] = vb;
            kcur[i] = __bfloat162float(kb);
            vcur[i] = __bfloat162float(vb);
        }
        float mx[GQ], l[GQ], acc[GQ][4];
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
            mx[hh] = -INFINITY; l[hh] = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[hh][i] = 0.f;
        }
        constexpr int U = 8;
        for (int j0 = 0; j0 <= pos; j0 += U) {
            float kr[U][4], vr[U][4];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = j0 + u;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (j < pos) {
                        kr[u][i] = __bfloat162float(Kc[base + (size_t)j * HD + lane + 32 * i]);
                        vr[u][i] = __bfloat162float(Vc[base + (size_t)j * HD + lane + 32 * i]);
                    } else {
                        kr[u][i] = kcur[i];
                        vr[u][i] = vcur[i];
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (j0 + u > pos) break;   // uniform over the warp (one token per warp)
#pragma unroll
                for (int hh = 0; hh < GQ; ++hh) {
                    const float sc = warp_sum(fmaf(q[hh][0], kr[u][0], fmaf(q[hh][1], kr[u][1],
                                                   fmaf(q[hh][2], kr[u][2], q[hh][3] * kr[u][3]))));
                    const float mn = fmaxf(mx[hh], sc);
                    const float cf = expf(mx[hh] - mn);
                    const float p = expf(sc - mn);
                    l[hh] = l[hh] * cf + p;
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[hh][i] = fmaf(p, vr[u][i], acc[hh][i] * cf);
                    mx[hh] = mn;
                }
            }
        }
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh)
#pragma unroll
            for (int i = 0; i < 4; ++i) res[hh][i] = acc[hh][i] / l[hh];
    } else if (pos >= 0 && lane == 0) {
        atomicOr(err, ERRB_BOUNDS);
    }
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const size_t o = (size_t)(g * GQ + hh) * HD + lane + 32 * i;
            if (hi) {
                const bf16 hv = __float2bfloat16_rn(res[hh][i]);
                hi[(size_t)m * nq * HD + o] = hv;
                lo[(size_t)m * nq * HD + o] = __float2bfloat16_rn(res[hh][i] - __bfloat162float(hv));
            } else {
                out[(size_t)m * ldo + o] = res[hh][i];
            }
        }
    }
}

cudaError_t launch_attention_short_fused(const float* qkv, int ldq, int M, int nq, int nkv, const float* q_norm,
                                         const float* k_norm, float eps, const float* rope_cs, int rope_rows,
                                         void* Kc, void* Vc, int cap, const int* tok_row, const int* tok_pos,
                                         float* out, int ldo, int* err, cudaStream_t st, const TcScratch* split) {
    if (M <= 0) return cudaSuccess;
    if (nq != 2 * nkv || cap > 64) return cudaErrorInvalidValue;
    bf16* hi = nullptr;
    bf16* lo = nullptr;
    if (split) {
        if (!tc_fits(*split, M, nq * HD)) return cudaErrorInvalidValue;
        hi = (bf16*)split->base;
        lo = hi + (size_t)M * nq * HD;
    }
    launch_pdl(attn_short_fused_kernel<2>, (M * nkv + 7) / 8, 256, 0, st, qkv, ldq, M, nq, nkv, q_norm, k_norm, eps,
               (const float2*)rope_cs, rope_rows, (bf16*)Kc, (bf16*)Vc, cap, tok_row, tok_pos, out, ldo, hi, lo, err);
    return cudaGetLastError();
}

template <int GQ>
static cudaError_t attention_bulk(const float* qkv, int ldq, int M, int nq, int nkv, const bf16* Kc, const bf16* Vc,
                                  int cap, const int* tok_row, const int* tok_pos, int n_splits, float* pm, float* pl,
                                  float* pacc, float* out, int ldo, bf16* hi, bf16* lo, int* err, cudaStream_t st) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(attn_bulk_kernel<GQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)ab::SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    launch_pdl(attn_bulk_kernel<GQ>, dim3(n_splits, nkv, M), ab::NT, ab::SMEM, st, qkv, ldq, nq, nkv, Kc, Vc, cap, tok_row,
                                                                          tok_pos, n_splits, pm, pl, pacc, out, ldo,
                                                                          hi, lo, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || n_splits == 1) return e;
    launch_pdl(attn_combine_kernel, dim3(M, nq), 128, 0, st, pm, pl, pacc, n_splits, nq, tok_pos, out, ldo, hi, lo);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t attention_impl(const float* qkv, int ldq, int M, int nq, int nkv, const T* Kc, const T* Vc, int cap,
                                  const int* tok_row, const int* tok_pos, int n_splits, float* pm, float* pl,
                                  float* pacc, float* out, int ldo, bf16* hi, bf16* lo, cudaStream_t st) {
    dim3 grid(n_splits, nkv, M);
    const int gq = nq / nkv;
    switch (gq) {
        case 1: launch_pdl(attn_split_kernel<T, 1>, grid, 128, 0, st, qkv, ldq, nq, nkv, Kc, Vc, cap, tok_row, tok_pos, n_splits, pm, pl, pacc); break;
        case 2: launch_pdl(attn_split_kernel<T, 2>, grid, 128, 0, st, qkv, ldq, nq, nkv, Kc, Vc, cap, tok_row, tok_pos, n_splits, pm, pl, pacc); break;
        case 4: launch_pdl(attn_split_kernel<T, 4>, grid, 128, 0, st, qkv, ldq, nq, nkv, Kc, Vc, cap, tok_row, tok_pos, n_splits, pm, pl, pacc); break;
        default: return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    launch_pdl(attn_combine_kernel, dim3(M, nq), 128, 0, st, pm, pl, pacc, n_splits, nq, tok_pos, out, ldo, hi, lo);
    return cudaGetLastError();
}

cudaError_t launch_attention(int dtype, const float* qkv, int ldq, int M, int nq, int nkv, const void* Kc,
                             const void* Vc, int cap, const int* tok_row, const int* tok_pos, int n_splits,
                             float* part_m, float* part_l, float* part_acc, float* out, int ldo, int* err,
                             cudaStream_t st, const TcScratch* split) {
    if (M <= 0) return cudaSuccess;
    bf16* hi = nullptr;
    bf16* lo = nullptr;
    if (split) {
        if (!tc_fits(*split, M, nq * HD)) return cudaErrorInvalidValue;
        hi = (bf16*)split->base;
        lo = hi + (size_t)M * nq * HD;
    }
    if (dtype == Q3_BF16 && nq == 2 * nkv && cap <= 64 && ldo % 4 == 0) {
        launch_pdl(attn_short_kernel<2>, (M * nkv + 7) / 8, 256, 0, st, qkv, ldq, M, nq, nkv, (const bf16*)Kc, (const bf16*)Vc,
                                                                cap, tok_row, tok_pos, out, ldo, hi, lo, err);
        return cudaGetLastError();
    }
    if (dtype == Q3_BF16 && nq == 2 * nkv)
        return attention_bulk<2>(qkv, ldq, M, nq, nkv, (const bf16*)Kc, (const bf16*)Vc, cap, tok_row, tok_pos,
                                 n_splits, part_m, part_l, part_acc, out, ldo, hi, lo, err, st);
    if (dtype == Q3_BF16)
        return attention_impl<bf16>(qkv, ldq, M, nq, nkv, (const bf16*)Kc, (const bf16*)Vc, cap, tok_row, tok_pos,
                                    n_splits, part_m, part_l, part_acc, out, ldo, hi, lo, st);
    return attention_impl<float>(qkv, ldq, M, nq, nkv, (const float*)Kc, (const float*)Vc, cap, tok_row, tok_pos,
                                 n_splits, part_m, part_l, part_acc, out, ldo, hi, lo, st);
}

}  // namespace q3

namespace q3 {

// ------------------------------------------------------------------ tiled causal prefill attention
// One block: 64 consecutive prompt tokens of one row (a query tile) and one
// KV head (its GQ = 2 q heads), over the row's cached positions 0..last.  K
// and V are staged in shared memory 64 positions at a time and read once for
// all 128 query rows (64 tokens x 2 heads).  Q Kt and P V run on the tensor
// cores (mma.m16n8k16, bf16 in, fp32 accumulate) with the fp32 operands Q and
// P as bf16 high + low parts, so the products keep fp32 accuracy; softmax is
// online (running max and sum per query row).  Warp w owns query rows
// 16 w .. 16 w + 15 (head w / 4, tokens 16 (w % 4) ..).
namespace pa {
constexpr int TQ = 64;          // tokens per query tile
constexpr int KB = 64;          // positions per K/V block
constexpr int KP = HD + 8;      // padded K row (bf16): fragment loads of 8 rows hit distinct banks
constexpr int VP = KB + 8;      // padded V^T row (bf16)

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return a | (b << 16);
}
// x = hi + lo in bf16 (two elements per register)
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& h, uint32_t& l) {
    const float h0 = __bfloat162float(__float2bfloat16_rn(x0)), h1 = __bfloat162float(__float2bfloat16_rn(x1));
    h = pack2(h0, h1);
    l = pack2(x0 - h0, x1 - h1);
}
__device__ __forceinline__ void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                    uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
}  // namespace pa

// tiles[t] = {first token m0, tokens n (1..64), row, position of token m0}
template <typename T>
__global__ void __launch_bounds__(256) prefill_attn_kernel(const float* __restrict__ qkv, int ldq, int nq, int nkv,
                                                           const T* __restrict__ Kc, const T* __restrict__ Vc,
                                                           int cap, const int4* __restrict__ tiles,
                                                           float* __restrict__ out, int ldo, bf16* __restrict__ ohi,
                                                           bf16* __restrict__ olo) {
    pdl_wait();
    pdl_trigger();
    using namespace pa;
    constexpr int GQ = 2;
    __shared__ __align__(16) bf16 sK[KB][KP];
    __shared__ __align__(16) bf16 sVt[HD][VP];
    const int4 tile = tiles[blockIdx.x];
    const int m0 = tile.x, ntok = tile.y, row = tile.z, p0 = tile.w;
    const int g = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, q4 = lane & 3;
    const int hh = warp >> 2;                 // q head within the group
    const int t0 = (warp & 3) * 16;           // first token of the warp's 16 query rows
    const int qh = g * GQ + hh;
    const float scale = 0.08838834764831845f; // 1/sqrt(128)

    // Q fragments (A operand of Q Kt): rows t0 + gq and t0 + gq + 8, high and low parts
    uint32_t qa[HD / 16][4], ql[HD / 16][4];
    {
        const int tr0 = min(t0 + gq, ntok - 1), tr1 = min(t0 + gq + 8, ntok - 1);
        const float* q0 = qkv + (size_t)(m0 + tr0) * ldq + (size_t)qh * HD;
        const float* q1 = qkv + (size_t)(m0 + tr1) * ldq + (size_t)qh * HD;
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
            const int d = ks * 16 + 2 * q4;
            split2(q0[d] * scale, q0[d + 1] * scale, qa[ks][0], ql[ks][0]);
            split2(q1[d] * scale, q1[d + 1] * scale, qa[ks][1], ql[ks][1]);
            split2(q0[d + 8] * scale, q0[d + 9] * scale, qa[ks][2], ql[ks][2]);
            split2(q1[d + 8] * scale, q1[d + 9] * scale, qa[ks][3], ql[ks][3]);
        }
    }
    // positions of this lane's two query rows
    const int pr0 = p0 + t0 + gq, pr1 = p0 + t0 + gq + 8;
    float o[HD / 8][4];
#pragma unroll
    for (int n = 0; n < HD / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float mx0 = -INFINITY, mx1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    const int last = p0 + ntok - 1;           // last position any query of the tile sees
    const size_t base = ((size_t)row * nkv + g) * cap * HD;
    for (int kb0 = 0; kb0 <= last; kb0 += KB) {
        const int nk = min(KB, last + 1 - kb0);
        __syncthreads();   // the previous block's K / V are no longer read
        // stage K [pos][dim] and V^T [dim][pos] (bf16); positions past nk are
        // zero.  K: consecutive threads take consecutive 8-dim pieces of a row
        // (16-byte stores, conflict-free); V: consecutive threads take
        // consecutive positions, so the transposed 2-byte stores of a warp hit
        // consecutive addresses of one V^T row.
        if constexpr (std::is_same<T, bf16>::value) {
            for (int i = tid; i < KB * (HD / 8); i += 256) {
                const int j = i / (HD / 8), c = (i % (HD / 8)) * 8;
                uint4 kv = make_uint4(0u, 0u, 0u, 0u);
                if (j < nk) kv = *reinterpret_cast<const uint4*>(Kc + base + (size_t)(kb0 + j) * HD + c);
                *reinterpret_cast<uint4*>(&sK[j][c]) = kv;
            }
            for (int i = tid; i < KB * (HD / 8); i += 256) {
                const int j = i % KB, c = (i / KB) * 8;
                uint4 vv = make_uint4(0u, 0u, 0u, 0u);
                if (j < nk) vv = *reinterpret_cast<const uint4*>(Vc + base + (size_t)(kb0 + j) * HD + c);
                const uint32_t w[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    sVt[c + 2 * e][j] = __ushort_as_bfloat16((unsigned short)(w[e] & 0xffffu));
                    sVt[c + 2 * e + 1][j] = __ushort_as_bfloat16((unsigned short)(w[e] >> 16));
                }
            }
        } else {
            for (int i = tid; i < KB * (HD / 8); i += 256) {
                const int j = i / (HD / 8), c = (i % (HD / 8)) * 8;
                float kv[8], vv[8];
                if (j < nk) {
                    load8(Kc + base + (size_t)(kb0 + j) * HD + c, kv);
                    load8(Vc + base + (size_t)(kb0 + j) * HD + c, vv);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) kv[e] = vv[e] = 0.f;
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    sK[j][c + e] = __float2bfloat16_rn(kv[e]);
                    sVt[c + e][j] = __float2bfloat16_rn(vv[e]);
                }
            }
        }
        __syncthreads();
        // S = Q Kt for the warp's 16 rows x 64 positions
        float sc[KB / 8][4];
#pragma unroll
        for (int n = 0; n < KB / 8; ++n) {
            sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
            const bf16* kr = &sK[n * 8 + gq][0];
#pragma unroll
            for (int ks = 0; ks < HD / 16; ++ks) {
                const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kr + ks * 16 + 2 * q4);
                const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kr + ks * 16 + 2 * q4 + 8);
                mma(sc[n], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
                mma(sc[n], ql[ks][0], ql[ks][1], ql[ks][2], ql[ks][3], b0, b1);
            }
        }
        // causal mask and online softmax: lane holds rows gq (c0, c1) and gq + 8 (c2, c3)
        float bm0 = -INFINITY, bm1 = -INFINITY;
#pragma unroll
        for (int n = 0; n < KB / 8; ++n) {
            const int j = kb0 + n * 8 + 2 * q4;
            if (j > pr0 || j - kb0 >= nk) sc[n][0] = -INFINITY;
            if (j + 1 > pr0 || j + 1 - kb0 >= nk) sc[n][1] = -INFINITY;
            if (j > pr1 || j - kb0 >= nk) sc[n][2] = -INFINITY;
            if (j + 1 > pr1 || j + 1 - kb0 >= nk) sc[n][3] = -INFINITY;
            bm0 = fmaxf(bm0, fmaxf(sc[n][0], sc[n][1]));
            bm1 = fmaxf(bm1, fmaxf(sc[n][2], sc[n][3]));
        }
        bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, 1));
        bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, 2));
        bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, 1));
        bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, 2));
        const float nm0 = fmaxf(mx0, bm0), nm1 = fmaxf(mx1, bm1);
        // rows with nothing visible yet keep a zero state (their max stays -inf)
        const float c0 = nm0 == -INFINITY ? 1.f : expf(mx0 - nm0);
        const float c1 = nm1 == -INFINITY ? 1.f : expf(mx1 - nm1);
        float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
        for (int n = 0; n < KB / 8; ++n) {
            sc[n][0] = nm0 == -INFINITY ? 0.f : expf(sc[n][0] - nm0);
            sc[n][1] = nm0 == -INFINITY ? 0.f : expf(sc[n][1] - nm0);
            sc[n][2] = nm1 == -INFINITY ? 0.f : expf(sc[n][2] - nm1);
            sc[n][3] = nm1 == -INFINITY ? 0.f : expf(sc[n][3] - nm1);
            rs0 += sc[n][0] + sc[n][1];
            rs1 += sc[n][2] + sc[n][3];
        }
        rs0 += __shfl_xor_sync(0xffffffffu, rs0, 1);
        rs0 += __shfl_xor_sync(0xffffffffu, rs0, 2);
        rs1 += __shfl_xor_sync(0xffffffffu, rs1, 1);
        rs1 += __shfl_xor_sync(0xffffffffu, rs1, 2);
        l0 = l0 * c0 + rs0;
        l1 = l1 * c1 + rs1;
        mx0 = nm0;
        mx1 = nm1;
#pragma unroll
        for (int n = 0; n < HD / 8; ++n) { o[n][0] *= c0; o[n][1] *= c0; o[n][2] *= c1; o[n][3] *= c1; }
        // O += P V: the S fragments of positions 16 k .. 16 k + 15 are the A fragment of step k
#pragma unroll
        for (int k = 0; k < KB / 16; ++k) {
            uint32_t ph[4], pl[4];
            split2(sc[2 * k][0], sc[2 * k][1], ph[0], pl[0]);
            split2(sc[2 * k][2], sc[2 * k][3], ph[1], pl[1]);
            split2(sc[2 * k + 1][0], sc[2 * k + 1][1], ph[2], pl[2]);
            split2(sc[2 * k + 1][2], sc[2 * k + 1][3], ph[3], pl[3]);
#pragma unroll
            for (int n = 0; n < HD / 8; ++n) {
                const bf16* vr = &sVt[n * 8 + gq][k * 16];
                const uint32_t b0 = *reinterpret_cast<const uint32_t*>(vr + 2 * q4);
                const uint32_t b1 = *reinterpret_cast<const uint32_t*>(vr + 2 * q4 + 8);
                mma(o[n], ph[0], ph[1], ph[2], ph[3], b0, b1);
                mma(o[n], pl[0], pl[1], pl[2], pl[3], b0, b1);
            }
        }
    }
    // normalise and store rows t0 + gq (c0, c1) and t0 + gq + 8 (c2, c3)
    const float i0 = 1.0f / l0, i1 = 1.0f / l1;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int tr = t0 + gq + 8 * hr;
        if (tr >= ntok) continue;
        const int m = m0 + tr;
        const float inv = hr ? i1 : i0;
#pragma unroll
        for (int n = 0; n < HD / 8; ++n) {
            const int d = n * 8 + 2 * q4;
            const float v0 = o[n][2 * hr] * inv, v1 = o[n][2 * hr + 1] * inv;
            const size_t col = (size_t)qh * HD + d;
            if (ohi) {
                const bf16 h0 = __float2bfloat16_rn(v0), h1 = __float2bfloat16_rn(v1);
                ohi[(size_t)m * nq * HD + col] = h0;
                ohi[(size_t)m * nq * HD + col + 1] = h1;
                olo[(size_t)m * nq * HD + col] = __float2bfloat16_rn(v0 - __bfloat162float(h0));
                olo[(size_t)m * nq * HD + col + 1] = __float2bfloat16_rn(v1 - __bfloat162float(h1));
            } else {
                out[(size_t)m * ldo + col] = v0;
                out[(size_t)m * ldo + col + 1] = v1;
            }
        }
    }
}

cudaError_t launch_prefill_attention(int dtype, const float* qkv, int ldq, int M, int nq, int nkv, const void* Kc,
                                     const void* Vc, int cap, const int4* tiles, int n_tiles, float* out, int ldo,
                                     cudaStream_t st, const TcScratch* split) {
    if (n_tiles <= 0) return cudaSuccess;
    if (nq != 2 * nkv) return cudaErrorInvalidValue;
    bf16* hi = nullptr;
    bf16* lo = nullptr;
    if (split) {
        if (!tc_fits(*split, M, nq * HD)) return cudaErrorInvalidValue;
        hi = (bf16*)split->base;
        lo = hi + (size_t)M * nq * HD;
    }
    dim3 grid(n_tiles, nkv);
    if (dtype == Q3_BF16)
        launch_pdl(prefill_attn_kernel<bf16>, grid, 256, 0, st, qkv, ldq, nq, nkv, (const bf16*)Kc, (const bf16*)Vc, cap,
                                                          tiles, out, ldo, hi, lo);
    else
        launch_pdl(prefill_attn_kernel<float>, grid, 256, 0, st, qkv, ldq, nq, nkv, (const float*)Kc, (const float*)Vc, cap,
                                                           tiles, out, ldo, hi, lo);
    return cudaGetLastError();
}

}  // namespace q3
