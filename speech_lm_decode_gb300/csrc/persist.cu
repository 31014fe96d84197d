// Persistent frame kernel: one talker step of a single row (code predictor
// 2-token prefill + 14 steps with their 15 draws, talker input assembly,
// 28-layer talker, codebook-0 selection) in ONE cooperative launch.
//
// Why: at batch 1 every projection is a GEMV that streams its weights once;
// the frame's ~3.3 GB (0.6B bf16) is bandwidth-trivial per phase (1-12 MB)
// but the phases are a ~550-long dependent chain.  Weights do not depend on
// activations, so each CTA's producer warp streams its slice of every
// upcoming projection into a shared-memory ring with bulk async copies
// (cp.async.bulk, completion on mbarriers) as far ahead as the ring allows,
// across phase boundaries.  The eight consumer warps only wait for the grid
// barrier that publishes the phase's input vector, then run the dot products
// out of shared memory.  HBM streaming therefore continues while the chain
// pays its barrier latencies.
//
// Layout of work: every GEMV phase splits its N output rows evenly over the
// CTAs (no split-K, fixed reduction order, no atomics on values).  Attention
// work items are (token, kv head, KV split); the last split of a head to
// finish merges the partials (flash-decoding combine).  Draws run on CTA 0.
//
// Every wait is bounded: an expired wait sets Q3's TIMEOUT error bit and the
// abort flag, which makes every other wait return; the producer then waits
// (bounded) for its own copies in flight before the CTA exits.
#include "sampler.cuh"
#include "kernels.h"
#include "frame_params.h"

#include <algorithm>

namespace q3 {

constexpr int NCW = 8;                       // consumer warps
constexpr int NTHREADS = (NCW + 1) * 32;     // + one producer warp
constexpr int TILE = 24 * 1024;              // bytes per ring slot
constexpr int NSLOT = 5;
constexpr long long WAIT_LIMIT = 4000000000LL;  // cycles (~2 s) before a wait gives up

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* b, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, unsigned bytes) {
    unsigned long long st;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 %0, [%1], %2;"
                 : "=l"(st) : "r"(smem_u32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    unsigned long long st;
    asm volatile("mbarrier.arrive.shared::cta.b64 %0, [%1];" : "=l"(st) : "r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, unsigned parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(b)), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* b) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 2, 256;" ::: "memory"); }

// activations written by other CTAs of this launch: read at L2, never from L1
__device__ __forceinline__ float ldg(const float* p) { return __ldcg(p); }
__device__ __forceinline__ int ldgi(const int* p) { return __ldcg(p); }
__device__ __forceinline__ float ld_kv(const bf16* p) { return __bfloat162float(__ldcg(p)); }
__device__ __forceinline__ float ld_kv(const float* p) { return __ldcg(p); }

// Wait on an mbarrier phase; false if the wait expired or the launch aborted.
__device__ bool mbar_wait(uint64_t* b, unsigned parity, const FrameParams& P) {
    if (mbar_try_wait(b, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(b, parity)) {
        if (*(volatile unsigned*)&P.bar[1]) return false;
        if (clock64() - t0 > WAIT_LIMIT) {
            atomicOr(P.err, ERRB_TIMEOUT);
            atomicExch(&P.bar[1], 1u);
            return false;
        }
    }
    return true;
}

// ------------------------------------------------------------------ shared memory
template <typename T>
struct FSmem {
    unsigned char ring[NSLOT][TILE];
    uint64_t full[NSLOT];
    uint64_t empty[NSLOT];
    float red[64];
    float resid[2][32];   // residual rows this CTA adds into (ADD epilogue), read in the prologue
    int flag;
    int aborted;
    // then: input vectors of the current GEMV phase, fp32 [2][kmax] (also the
    // attention phase's scratch); then the draw's scratch (CTA 0 only)
};

__host__ __device__ constexpr size_t align128(size_t v) { return (v + 127) & ~(size_t)127; }
template <typename T>
__device__ __forceinline__ float* xin_ptr(FSmem<T>& s) {
    return reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(&s) + align128(sizeof(FSmem<T>)));
}
template <typename T>
__device__ __forceinline__ SampSmem& samp_ptr(FSmem<T>& s, int xin_bytes) {
    const size_t off = align128(sizeof(FSmem<T>)) + align128((size_t)xin_bytes);
    return *reinterpret_cast<SampSmem*>(reinterpret_cast<unsigned char*>(&s) + off);
}

// ------------------------------------------------------------------ the frame schedule
// Both roles walk the same schedule; the producer acts on GEMV phases only.
// prologue: NORM = rmsnorm(vector) * w; LOAD = copy operand rows; RAW = operand of the raw vector
enum class Pro { NORM, LOAD, RAW };
// where the vector comes from: the residual rows (NONE) or an assembled token, whose
// residual slice this CTA also writes
enum class Tok { NONE, CP0, CPS, TALK };
enum class Epi { STORE, ADD, BIAS, GATED };

struct Gemv {
    const void* W;
    int N, K;
    bool gated;   // W holds [2N][K]: gate rows then up rows; output silu(g)*u
    int M;        // input vectors
    Pro pro;
    Tok tok;
    Epi epi;
    const float* pro_src;   // NORM: residual rows; LOAD: operand rows
    int pro_ld;
    const float* norm_w;
    float* dst;
    int ld_dst;
    const float* bias;
    float* hout;            // NORM: also write the fp32 normed vector (talker h)
    int s_idx;              // TOK_CPS: predictor step
};

__device__ __forceinline__ void split_rows(int N, int& n0, int& n1) {
    n0 = (int)(((long long)N * blockIdx.x) / gridDim.x);
    n1 = (int)(((long long)N * (blockIdx.x + 1)) / gridDim.x);
}

template <typename T>
__device__ __forceinline__ int rows_per_tile(const Gemv& g) {
    const int unit = g.K * (int)sizeof(T) * (g.gated ? 2 : 1);
    return max(1, TILE / unit);
}

// Cached positions [j0, j1) of a talker attention item that the producer
// prefetches (all before the new token's position p0); false if none, or if
// they do not fit one ring slot (then the consumer reads them directly).
template <typename T>
__device__ __forceinline__ bool kv_prefetch_range(const FrameParams& P, const PBlk& B, int M, int p0, int S, int item,
                                                  int& j0, int& j1) {
    const int m = item / (P.nkv * S);
    const int sp = item % S;
    const int n = p0 + m + 1;
    const int chunk = (n + S - 1) / S;
    j0 = sp * chunk;
    j1 = min(min(n, j0 + chunk), p0);
    return j1 > j0 && (size_t)(j1 - j0) * HD * sizeof(T) * 2 <= (size_t)TILE;
}

// ------------------------------------------------------------------ producer
template <typename T>
struct Producer {
    FSmem<T>& s;
    const FrameParams& P;
    unsigned seq = 0;
    bool ok = true;

    __device__ void gemv(const Gemv& g) {
        if (!ok) return;
        int n0, n1;
        split_rows(g.N, n0, n1);
        const int rt = rows_per_tile<T>(g);
        const size_t row_bytes = (size_t)g.K * sizeof(T);
        for (int r0 = n0; r0 < n1; r0 += rt) {
            const int r = min(rt, n1 - r0);
            const int slot = seq % NSLOT;
            const unsigned round = seq / NSLOT;
            if (round > 0 && !mbar_wait(&s.empty[slot], (round - 1) & 1, P)) { ok = false; return; }
            const unsigned bytes = (unsigned)(r * row_bytes * (g.gated ? 2 : 1));
            mbar_expect_tx(&s.full[slot], bytes);
            const char* src = (const char*)g.W + (size_t)r0 * row_bytes;
            bulk_g2s(s.ring[slot], src, (unsigned)(r * row_bytes), &s.full[slot]);
            if (g.gated)
                bulk_g2s(s.ring[slot] + r * row_bytes, (const char*)g.W + (size_t)(g.N + r0) * row_bytes,
                         (unsigned)(r * row_bytes), &s.full[slot]);
            ++seq;
        }
    }
    __device__ void barrier() {}
    // Talker attention: the cached K / V of positions before the new token do
    // not depend on this step; stream each of this CTA's splits into a slot.
    __device__ void attention(int l, const PBlk& B, int M, int p0, int S, bool talker) {
        if (!ok || !talker) return;
        for (int item = blockIdx.x; item < M * P.nkv * S; item += gridDim.x) {
            int j0, j1;
            if (!kv_prefetch_range<T>(P, B, M, p0, S, item, j0, j1)) continue;
            const int g = (item / S) % P.nkv;
            const int slot = seq % NSLOT;
            const unsigned round = seq / NSLOT;
            if (round > 0 && !mbar_wait(&s.empty[slot], (round - 1) & 1, P)) { ok = false; return; }
            const size_t row_bytes = (size_t)HD * sizeof(T);
            const size_t base = (((size_t)l * P.max_batch + 0) * P.nkv + g) * B.cap + j0;
            const unsigned bytes = (unsigned)((j1 - j0) * row_bytes);
            mbar_expect_tx(&s.full[slot], 2 * bytes);
            bulk_g2s(s.ring[slot], (const char*)B.Kc + base * row_bytes, bytes, &s.full[slot]);
            bulk_g2s(s.ring[slot] + bytes, (const char*)B.Vc + base * row_bytes, bytes, &s.full[slot]);
            ++seq;
        }
    }
    __device__ void sample_cp(int) {}
    __device__ void sample_talker() {}
    __device__ void prepare_talker() {}
    __device__ int talker_pos() const { return pos; }
    int pos = 0;
    __device__ bool live() const { return ok; }

    // copies issued but not yet consumed must land before the CTA exits
    __device__ void drain() {
        for (unsigned t = (seq > NSLOT ? seq - NSLOT : 0); t < seq; ++t) {
            const long long t0 = clock64();
            while (!mbar_try_wait(&s.full[t % NSLOT], (t / NSLOT) & 1))
                if (clock64() - t0 > WAIT_LIMIT) break;
        }
    }
};

// ------------------------------------------------------------------ consumer
template <typename T, int GQ>
struct Consumer {
    FSmem<T>& s;
    const FrameParams& P;
    unsigned seq = 0;
    unsigned epoch = 0;
    int frame = 0;      // frame completed by this step
    int pos = 0;        // talker position of the new token
    bool ok = true;

    __device__ float* xin() { return xin_ptr<T>(s); }

    __device__ float block_sum(float v) {
        v = warp_sum(v);
        const int w = threadIdx.x >> 5;
        consumer_sync();
        if ((threadIdx.x & 31) == 0) s.red[w] = v;
        consumer_sync();
        float r = 0.f;
#pragma unroll
        for (int i = 0; i < NCW; ++i) r += s.red[i];
        return r;
    }

    __device__ void abort_now() {
        atomicExch(&P.bar[1], 1u);
        ok = false;
    }

    // Grid-wide barrier: publish this CTA's writes of the phase, wait for all CTAs.
    __device__ void barrier() {
        consumer_sync();
        ++epoch;
        if (threadIdx.x == 0) {
            int ab = 0;
            if (ok) {
                __threadfence();
                atomicAdd(&P.bar[0], 1u);
                const unsigned target = epoch * gridDim.x;
                const long long t0 = clock64();
                while (ld_acquire(&P.bar[0]) < target) {
                    if (*(volatile unsigned*)&P.bar[1]) { ab = 1; break; }
                    if (clock64() - t0 > WAIT_LIMIT) {
                        atomicOr(P.err, ERRB_TIMEOUT);
                        atomicExch(&P.bar[1], 1u);
                        ab = 1;
                        break;
                    }
                }
            } else {
                ab = 1;
            }
            s.aborted = ab;
        }
        consumer_sync();
        if (s.aborted) ok = false;
    }

    __device__ bool live() const { return ok; }

    // ---------------- token vectors (talker width H) for prologues
    // Sources of the input vectors of a phase, resolved once per phase.
    struct Src {
        const float* f32;   // fp32 vector (residual rows, h) read at L2
        const T* tab;       // embedding table row
    };
    __device__ Src source(const Gemv& g, int m) {
        Src r{nullptr, nullptr};
        const int H = P.H;
        if (g.tok == Tok::NONE) {
            r.f32 = g.pro_src + (size_t)m * g.pro_ld;
        } else if (g.tok == Tok::CP0) {
            if (m == 0) r.f32 = P.h;
            else r.tab = (const T*)P.codec_emb + (size_t)P.rows[0].code0 * H;
        } else if (g.tok == Tok::CPS) {
            const int c = ldgi(P.codes + ((size_t)frame * MAX_GROUPS + g.s_idx));
            if (c < 0 || c >= P.cpV) {
                if (threadIdx.x == 0) atomicOr(P.err, ERRB_BOUNDS);
                abort_now();
                r.tab = (const T*)P.cp_emb;
            } else {
                r.tab = (const T*)P.cp_emb + ((size_t)(g.s_idx - 1) * P.cpV + c) * H;
            }
        }
        return r;
    }
    __device__ float value(const Gemv& g, const Src& src, int i) {
        if (g.tok == Tok::TALK) return talker_input(i);
        return src.f32 ? ldg(src.f32 + i) : to_f(src.tab[i]);
    }

    // input vectors of a GEMV phase -> shared memory (fp32), one pass over
    // global memory; ADD phases also fetch the residual rows they update
    __device__ void prologue(const Gemv& g) {
        float* xs = xin();
        const int K = g.K;
        const int tid = threadIdx.x;
        if (g.epi == Epi::ADD) {
            int n0, n1;
            split_rows(g.N, n0, n1);
            for (int i = tid; i < g.M * 32; i += 256) {
                const int m = i / 32, r = i % 32;
                if (n0 + r < n1) s.resid[m][r] = ldg(g.dst + (size_t)m * g.ld_dst + n0 + r);
            }
        }
        if (g.pro == Pro::LOAD) {
            for (int m = 0; m < g.M; ++m)
                for (int i = tid; i < K; i += 256) xs[m * K + i] = ldg(g.pro_src + (size_t)m * g.pro_ld + i);
            consumer_sync();
            return;
        }
        if (g.pro == Pro::RAW) {   // predictor tokens into the width projection
            for (int m = 0; m < g.M; ++m) {
                const Src src = source(g, m);
                for (int i = tid; i < K; i += 256) xs[m * K + i] = value(g, src, i);
            }
            consumer_sync();
            return;
        }
        // NORM: (token -> this CTA's residual slice) -> rmsnorm * w
        int r0, r1;
        split_rows(K, r0, r1);
        for (int m = 0; m < g.M; ++m) {
            const Src src = source(g, m);
            float* resid = const_cast<float*>(g.pro_src) + (size_t)m * g.pro_ld;
            float ss = 0.f;
            for (int i = tid; i < K; i += 256) {
                const float v = value(g, src, i);
                xs[m * K + i] = v;
                ss = fmaf(v, v, ss);
                if (g.tok != Tok::NONE && i >= r0 && i < r1) resid[i] = v;
            }
            const float tot = block_sum(ss);
            const float r = 1.0f / sqrtf(tot / (float)K + P.eps);
            for (int i = tid; i < K; i += 256) {
                const float v = xs[m * K + i] * r * g.norm_w[i];
                xs[m * K + i] = v;
                if (g.hout && i >= r0 && i < r1) g.hout[i] = v;
            }
        }
        consumer_sync();
    }

    // talker input (A1): codec_emb(code0) + sum_q table[q-1](code_q) + text row
    int tk_ids[MAX_GROUPS];
    const float* tk_text = nullptr;
    __device__ void prepare_talker() {
        if (!ok) return;
        const RowState& rs = P.rows[0];
        bool good = true;
        for (int q = 0; q < P.G; ++q) {
            tk_ids[q] = ldgi(P.codes + ((size_t)frame * MAX_GROUPS + q));
            good &= tk_ids[q] >= 0 && tk_ids[q] < (q == 0 ? P.V : P.cpV);
        }
        if (!good) {
            if (threadIdx.x == 0) atomicOr(P.err, ERRB_BOUNDS);
            abort_now();
            for (int q = 0; q < P.G; ++q) tk_ids[q] = 0;
        }
        tk_text = frame < rs.n_text ? P.text + (size_t)(rs.text_off + frame) * P.H : P.pad;
    }
    __device__ int talker_pos() const { return pos; }
    __device__ float talker_input(int i) {
        const int H = P.H;
        float acc = to_f(((const T*)P.codec_emb)[(size_t)tk_ids[0] * H + i]);
        for (int q = 1; q < P.G; ++q) acc += to_f(((const T*)P.cp_emb)[((size_t)(q - 1) * P.cpV + tk_ids[q]) * H + i]);
        return acc + tk_text[i];
    }

    template <int M, bool GATED>
    __device__ void gemv_tiles(const Gemv& g) {
        int n0, n1;
        split_rows(g.N, n0, n1);
        const int rt = rows_per_tile<T>(g);
        const int K = g.K;
        const size_t row_bytes = (size_t)K * sizeof(T);
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const float* xs = xin();
        for (int r0 = n0; r0 < n1; r0 += rt) {
            const int r = min(rt, n1 - r0);
            const int slot = seq % NSLOT;
            const unsigned round = seq / NSLOT;
            ++seq;
            if (!mbar_wait(&s.full[slot], round & 1, P)) { ok = false; return; }
            const unsigned char* tile = s.ring[slot];
            for (int i = warp; i < r; i += NCW) {
                const T* wr = (const T*)(tile + i * row_bytes);
                const T* ur = (const T*)(tile + (r + i) * row_bytes);
                float acc[M], accu[M];
#pragma unroll
                for (int m = 0; m < M; ++m) { acc[m] = 0.f; accu[m] = 0.f; }
                for (int k = lane * 8; k < K; k += 256) {
                    float w[8], u[8];
                    load8(wr + k, w);
                    if (GATED) load8(ur + k, u);
#pragma unroll
                    for (int m = 0; m < M; ++m) {
                        float xv[8];
                        load8(xs + m * K + k, xv);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            acc[m] = fmaf(w[j], xv[j], acc[m]);
                            if (GATED) accu[m] = fmaf(u[j], xv[j], accu[m]);
                        }
                    }
                }
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    const float v = warp_sum(acc[m]);
                    const float uu = GATED ? warp_sum(accu[m]) : 0.f;
                    if (lane == 0) {
                        const int n = r0 + i;
                        float* d = g.dst + (size_t)m * g.ld_dst + n;
                        if (GATED) {
                            *d = v / (1.0f + expf(-v)) * uu;
                        } else if (g.epi == Epi::ADD) {
                            *d = s.resid[m][n - n0] + v;
                        } else if (g.epi == Epi::BIAS) {
                            *d = v + g.bias[n];
                        } else {
                            *d = v;
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.empty[slot]);
        }
    }

    __device__ void gemv(const Gemv& g) {
        if (!ok) return;
        prologue(g);
        if (!ok) return;
        if (g.gated) {
            if (g.M == 1) gemv_tiles<1, true>(g); else gemv_tiles<2, true>(g);
        } else {
            if (g.M == 1) gemv_tiles<1, false>(g); else gemv_tiles<2, false>(g);
        }
    }

    // ---------------- attention (A4 + A5) for M new tokens at positions p0.. of a layer
    // smem use: the xin region (not needed during this phase): q [GQ][HD], k/v of new tokens [2][HD] each.
    __device__ void attention(int l, const PBlk& B, int M, int p0, int S, bool talker) {
        if (!ok) return;
        const int nq = P.nq, nkv = P.nkv;
        const int nqkv = (nq + 2 * nkv) * HD;
        const int items = M * nkv * S;
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        float* sq = reinterpret_cast<float*>(xin());       // [GQ][HD]
        float* sk = sq + GQ * HD;                          // [2][HD] new keys (rounded as cached)
        float* sv = sk + 2 * HD;                           // [2][HD] new values
        float* sm_m = sv + 2 * HD;                         // [NCW][GQ]
        float* sm_l = sm_m + NCW * GQ;                     // [NCW][GQ]
        float* sacc = sm_l + NCW * GQ;                     // [NCW][GQ][HD]
        for (int item = blockIdx.x; item < items; item += gridDim.x) {
            const int m = item / (nkv * S);
            const int g = (item / S) % nkv;
            const int sp = item % S;
            const int pos = p0 + m;
            const int n = pos + 1;
            const int chunk = (n + S - 1) / S;
            const int j0 = sp * chunk, j1 = min(n, j0 + chunk);
            // cache [L][max_batch][nkv][cap][HD], row 0
            T* Kg = (T*)B.Kc + (((size_t)l * P.max_batch + 0) * nkv + g) * B.cap * HD;
            T* Vg = (T*)B.Vc + (((size_t)l * P.max_batch + 0) * nkv + g) * B.cap * HD;
            // q heads of this group (token m), k/v of the new tokens 0..m: QK-norm + RoPE
            const int tasks = GQ + 2 * (m + 1);
            for (int t = warp; t < tasks; t += NCW) {
                const float* src;
                float* dst;
                const float* wn = nullptr;
                int tp;       // position for RoPE
                bool rope = true;
                if (t < GQ) {
                    src = P.qkv + (size_t)m * nqkv + (size_t)(g * GQ + t) * HD;
                    dst = sq + t * HD; wn = B.q_norm + (size_t)l * HD; tp = pos;
                } else if (t < GQ + m + 1) {
                    const int mm = t - GQ;
                    src = P.qkv + (size_t)mm * nqkv + (size_t)(nq + g) * HD;
                    dst = sk + mm * HD; wn = B.k_norm + (size_t)l * HD; tp = p0 + mm;
                } else {
                    const int mm = t - GQ - (m + 1);
                    src = P.qkv + (size_t)mm * nqkv + (size_t)(nq + nkv + g) * HD;
                    dst = sv + mm * HD; rope = false; tp = 0;
                }
                float e[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) e[i] = ldg(src + lane + 32 * i);
                if (rope) {
                    const float ss = warp_sum(e[0] * e[0] + e[1] * e[1] + e[2] * e[2] + e[3] * e[3]);
                    const float r = 1.0f / sqrtf(ss / (float)HD + P.eps);
#pragma unroll
                    for (int i = 0; i < 4; ++i) e[i] = e[i] * r * wn[lane + 32 * i];
                    const float2 c0 = P.rope[(size_t)tp * (HD / 2) + lane];
                    const float2 c1 = P.rope[(size_t)tp * (HD / 2) + lane + 32];
                    float a = e[0], b = e[2];
                    e[0] = a * c0.x - b * c0.y; e[2] = b * c0.x + a * c0.y;
                    a = e[1]; b = e[3];
                    e[1] = a * c1.x - b * c1.y; e[3] = b * c1.x + a * c1.y;
                }
                const bool is_kv = t >= GQ;
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[lane + 32 * i] = is_kv ? to_f(from_f<T>(e[i])) : e[i];
            }
            consumer_sync();
            // the split holding this token's own position appends its k / v to the cache
            if (pos >= j0 && pos < j1) {
                for (int i = threadIdx.x; i < HD; i += 256) {
                    Kg[(size_t)pos * HD + i] = from_f<T>(sk[m * HD + i]);
                    Vg[(size_t)pos * HD + i] = from_f<T>(sv[m * HD + i]);
                }
            }
            // cached positions of a talker split come from the ring (prefetched)
            const T* kring = nullptr;
            const T* vring = nullptr;
            int pj0 = 0, pj1 = 0, slot = -1;
            if (talker && kv_prefetch_range<T>(P, B, M, p0, S, item, pj0, pj1)) {
                slot = seq % NSLOT;
                const unsigned round = seq / NSLOT;
                ++seq;
                if (!mbar_wait(&s.full[slot], round & 1, P)) { ok = false; }
                kring = (const T*)s.ring[slot];
                vring = kring + (size_t)(pj1 - pj0) * HD;
            }
            // online softmax over positions j0..j1-1, one position per warp step
            float mx[GQ], lsum[GQ], acc[GQ][4];
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) {
                mx[hh] = -INFINITY; lsum[hh] = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[hh][i] = 0.f;
            }
            const float scale = 0.08838834764831845f;
            for (int j = j0 + warp; j < j1; j += NCW) {
                float kk[4], vv[4];
                if (kring && j >= pj0 && j < pj1) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        kk[i] = to_f(kring[(size_t)(j - pj0) * HD + lane + 32 * i]);
                        vv[i] = to_f(vring[(size_t)(j - pj0) * HD + lane + 32 * i]);
                    }
                } else if (j < p0) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        kk[i] = ld_kv(Kg + (size_t)j * HD + lane + 32 * i);
                        vv[i] = ld_kv(Vg + (size_t)j * HD + lane + 32 * i);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        kk[i] = sk[(j - p0) * HD + lane + 32 * i];
                        vv[i] = sv[(j - p0) * HD + lane + 32 * i];
                    }
                }
#pragma unroll
                for (int hh = 0; hh < GQ; ++hh) {
                    float d = 0.f;
#pragma unroll
                    for (int i = 0; i < 4; ++i) d = fmaf(sq[hh * HD + lane + 32 * i], kk[i], d);
                    d = warp_sum(d) * scale;
                    const float mn = fmaxf(mx[hh], d);
                    const float c = expf(mx[hh] - mn);
                    const float p = expf(d - mn);
                    lsum[hh] = lsum[hh] * c + p;
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[hh][i] = fmaf(p, vv[i], acc[hh][i] * c);
                    mx[hh] = mn;
                }
            }
            __syncwarp();
            if (slot >= 0 && lane == 0) mbar_arrive(&s.empty[slot]);
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) {
                if (lane == 0) { sm_m[warp * GQ + hh] = mx[hh]; sm_l[warp * GQ + hh] = lsum[hh]; }
#pragma unroll
                for (int i = 0; i < 4; ++i) sacc[(warp * GQ + hh) * HD + lane + 32 * i] = acc[hh][i];
            }
            consumer_sync();
            // merge the warps -> this split's partial
            float* part = P.part + ((((size_t)m * nkv + g) * S + sp) * GQ) * (HD + 2);
            for (int idx = threadIdx.x; idx < GQ * HD; idx += 256) {
                const int hh = idx / HD, d = idx % HD;
                float ma = -INFINITY;
                for (int w = 0; w < NCW; ++w) ma = fmaxf(ma, sm_m[w * GQ + hh]);
                float a = 0.f, ls = 0.f;
                for (int w = 0; w < NCW; ++w) {
                    const float c = (ma == -INFINITY) ? 0.f : expf(sm_m[w * GQ + hh] - ma);
                    a += sacc[(w * GQ + hh) * HD + d] * c;
                    ls += sm_l[w * GQ + hh] * c;
                }
                part[hh * (HD + 2) + d] = a;
                if (d == 0) { part[hh * (HD + 2) + HD] = ma; part[hh * (HD + 2) + HD + 1] = ls; }
            }
            // the last split of this (token, head group) to finish merges all splits
            consumer_sync();
            if (threadIdx.x == 0) {
                __threadfence();
                const unsigned old = atomicAdd(&P.bar[2 + m * nkv + g], 1u);
                s.flag = (old == (unsigned)S - 1);
            }
            consumer_sync();
            if (s.flag) {
                __threadfence();
                const float* pb = P.part + (((size_t)m * nkv + g) * S) * GQ * (HD + 2);
                for (int idx = threadIdx.x; idx < GQ * HD; idx += 256) {
                    const int hh = idx / HD, d = idx % HD;
                    float ma = -INFINITY;
                    for (int q = 0; q < S; ++q) ma = fmaxf(ma, ldg(pb + ((size_t)q * GQ + hh) * (HD + 2) + HD));
                    float num = 0.f, den = 0.f;
                    for (int q = 0; q < S; ++q) {
                        const float* pq = pb + ((size_t)q * GQ + hh) * (HD + 2);
                        const float mq = ldg(pq + HD);
                        const float c = (mq == -INFINITY) ? 0.f : expf(mq - ma);
                        num += ldg(pq + d) * c;
                        den += ldg(pq + HD + 1) * c;
                    }
                    P.o[(size_t)m * nq * HD + (size_t)(g * GQ + hh) * HD + d] = num / den;
                }
                if (threadIdx.x == 0) P.bar[2 + m * nkv + g] = 0u;
            }
            consumer_sync();
        }
    }

    // ---------------- draws on CTA 0
    __device__ void sample_cp(int sidx) {
        if (!ok || blockIdx.x != 0) return;
        SampSmem& sm = samp_ptr<T>(s, P.xin_bytes);
        const q3tts_sampling p = P.P[0];
        if (P.cap_c && P.cap_slot[0] >= 0 && frame < P.cap_T) {
            float* dst = P.cap_c + (((size_t)P.cap_slot[0] * P.cap_T + frame) * (P.G - 1) + sidx) * P.cpV;
            for (int i = threadIdx.x; i < P.cpV; i += 256) dst[i] = ldg(P.cpl + i);
        }
        const DrawCfg d{p.cp_do_sample, p.cp_temperature, p.cp_top_k, p.cp_top_p};
        const int id = sample_row(sm, P.cpl, P.cpV, d, false, 1.0f, nullptr, nullptr, 0, 0, -1, 0, 0, p.seed, 0u,
                                  (uint32_t)frame, (uint32_t)(sidx + 1));
        if (threadIdx.x == 0) {
            if (id < 0) {
                atomicOr(P.err, ERRB_NAN);
                RowState& rs = P.rows[0];
                rs.finished = 1;
                rs.reason = Q3_FINISHED_ERROR;
                rs.frames = frame;
                atomicExch(&P.bar[1], 1u);
            } else {
                P.codes[(size_t)frame * MAX_GROUPS + sidx + 1] = id;
            }
        }
    }

    __device__ void sample_talker() {
        if (!ok || blockIdx.x != 0) return;
        SampSmem& sm = samp_ptr<T>(s, P.xin_bytes);
        RowState& rs = P.rows[0];
        const q3tts_sampling p = P.P[0];
        const int k = frame + 1;
        if (P.cap_t && P.cap_slot[0] >= 0 && k <= P.cap_T) {
            float* dst = P.cap_t + ((size_t)P.cap_slot[0] * (P.cap_T + 1) + k) * P.V;
            for (int i = threadIdx.x; i < P.V; i += 256) dst[i] = ldg(P.logits + i);
        }
        const DrawCfg d{p.do_sample, p.temperature, p.top_k, p.top_p};
        int id = sample_row(sm, P.logits, P.V, d, true, p.repetition_penalty, rs.seen, nullptr, k, p.min_new_tokens,
                            P.eos, P.sup_lo, P.sup_hi, p.seed, 0u, (uint32_t)k, 0u);
        if (threadIdx.x == 0) {
            rs.frames = k;
            if (id < 0) {
                atomicOr(P.err, ERRB_NAN);
                rs.finished = 1;
                rs.reason = Q3_FINISHED_ERROR;
            } else {
                if (p.force_eos_at_frame >= 0 && k == p.force_eos_at_frame) id = P.eos;
                if (id < MAX_VOCAB) rs.seen[id >> 5] |= 1u << (id & 31);
                rs.code0 = id;
                rs.sel = k + 1;
                rs.pos += 1;
                if (id == P.eos) { rs.finished = 1; rs.reason = Q3_FINISHED_EOS; }
                else if (k >= p.max_frames) { rs.finished = 1; rs.reason = Q3_FINISHED_LENGTH; }
            }
        }
    }
};


// ------------------------------------------------------------------ schedule
template <typename T, class R>
__device__ void gemv_phase(R& r, const Gemv& g) {
    r.gemv(g);
    r.barrier();
}

template <typename T, class R>
__device__ void layer(R& r, const FrameParams& P, const PBlk& B, int l, int M, int p0, int S, float* x, Tok tok,
                      int s_idx, bool talker) {
    const size_t e = sizeof(T);
    const int nq = P.nq, nkv = P.nkv, H = B.H, F = B.F;
    const int nqkv = (nq + 2 * nkv) * HD;
    Gemv g{};
    // A2 + A3: (token assembly) + RMSNorm + q/k/v projection
    g.W = (const char*)B.wqkv + (size_t)l * nqkv * H * e; g.N = nqkv; g.K = H; g.M = M;
    g.pro = Pro::NORM; g.tok = tok; g.epi = Epi::STORE; g.pro_src = x; g.pro_ld = H;
    g.norm_w = B.attn_norm + (size_t)l * H; g.dst = P.qkv; g.ld_dst = nqkv; g.s_idx = s_idx;
    gemv_phase<T>(r, g);
    // A4 + A5
    r.attention(l, B, M, p0, S, talker);
    r.barrier();
    // A6: O projection + residual
    g = Gemv{};
    g.W = (const char*)B.wo + (size_t)l * H * nq * HD * e; g.N = H; g.K = nq * HD; g.M = M;
    g.pro = Pro::LOAD; g.tok = Tok::NONE; g.epi = Epi::ADD; g.pro_src = P.o; g.pro_ld = nq * HD;
    g.dst = x; g.ld_dst = H;
    gemv_phase<T>(r, g);
    // A7: RMSNorm + gate/up + SiLU(g)*u
    g = Gemv{};
    g.W = (const char*)B.wgu + (size_t)l * 2 * F * H * e; g.N = F; g.K = H; g.M = M; g.gated = true;
    g.pro = Pro::NORM; g.tok = Tok::NONE; g.epi = Epi::GATED; g.pro_src = x; g.pro_ld = H;
    g.norm_w = B.mlp_norm + (size_t)l * H; g.dst = P.act; g.ld_dst = F;
    gemv_phase<T>(r, g);
    // A8: down projection + residual
    g = Gemv{};
    g.W = (const char*)B.wd + (size_t)l * H * F * e; g.N = H; g.K = F; g.M = M;
    g.pro = Pro::LOAD; g.tok = Tok::NONE; g.epi = Epi::ADD; g.pro_src = P.act; g.pro_ld = F;
    g.dst = x; g.ld_dst = H;
    gemv_phase<T>(r, g);
}

template <typename T, class R>
__device__ void frame_schedule(R& r, const FrameParams& P) {
    const size_t e = sizeof(T);
    const int G1 = P.G - 1;
    const bool proj = P.H != P.Hc;
    // code predictor: tokens [h, codec_emb(code0)] at 0,1, then table[s-1](code_s) at s+1
    for (int s = 0; s < G1 && r.live(); ++s) {
        const int M = s == 0 ? 2 : 1;
        const Tok tok = s == 0 ? Tok::CP0 : Tok::CPS;
        Tok layer_tok = tok;
        if (proj) {
            Gemv g{};
            g.W = P.cp_proj_w; g.N = P.Hc; g.K = P.H; g.M = M; g.pro = Pro::RAW; g.tok = tok; g.epi = Epi::BIAS;
            g.bias = P.cp_proj_b; g.dst = P.cx; g.ld_dst = P.Hc; g.s_idx = s;
            gemv_phase<T>(r, g);
            layer_tok = Tok::NONE;
        }
        for (int l = 0; l < P.c.L && r.live(); ++l)
            layer<T>(r, P, P.c, l, M, 0 + (s == 0 ? 0 : s + 1), 1, P.cx, l == 0 ? layer_tok : Tok::NONE, s, false);
        // final norm of the last token -> head[s]
        Gemv g{};
        g.W = (const char*)P.cp_heads + (size_t)s * P.cpV * P.Hc * e; g.N = P.cpV; g.K = P.Hc; g.M = 1;
        g.pro = Pro::NORM; g.tok = Tok::NONE; g.epi = Epi::STORE; g.pro_src = P.cx + (size_t)(M - 1) * P.Hc;
        g.pro_ld = P.Hc; g.norm_w = P.c.final_norm; g.dst = P.cpl; g.ld_dst = P.cpV;
        gemv_phase<T>(r, g);
        r.sample_cp(s);
        r.barrier();
    }
    // talker
    r.prepare_talker();
    for (int l = 0; l < P.t.L && r.live(); ++l)
        layer<T>(r, P, P.t, l, 1, r.talker_pos(), P.n_splits, P.x, l == 0 ? Tok::TALK : Tok::NONE, 0, true);
    Gemv g{};
    g.W = P.codec_head; g.N = P.V; g.K = P.H; g.M = 1; g.pro = Pro::NORM; g.tok = Tok::NONE; g.epi = Epi::STORE;
    g.pro_src = P.x; g.pro_ld = P.H; g.norm_w = P.t.final_norm; g.dst = P.logits; g.ld_dst = P.V; g.hout = P.h;
    gemv_phase<T>(r, g);
    r.sample_talker();
}

template <typename T, int GQ>
__global__ void __launch_bounds__(NTHREADS, 1) frame_kernel(const FrameParams* __restrict__ Pp) {
    extern __shared__ __align__(128) unsigned char smraw[];
    FSmem<T>& s = *reinterpret_cast<FSmem<T>*>(smraw);
    const FrameParams& P = *Pp;
    if (P.rows[0].finished) return;   // uniform over the grid
    if (threadIdx.x == 0) {
        for (int i = 0; i < NSLOT; ++i) { mbar_init(&s.full[i], 1); mbar_init(&s.empty[i], NCW); }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s.aborted = 0;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    if (warp == NCW) {
        if ((threadIdx.x & 31) == 0) {
            Producer<T> pr{s, P};
            pr.pos = P.rows[0].pos;
            frame_schedule<T>(pr, P);
            pr.drain();
        }
        return;
    }
    Consumer<T, GQ> c{s, P};
    c.frame = P.rows[0].sel - 1;
    c.pos = P.rows[0].pos;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (c.frame < 0 || c.frame >= P.frames_cap || P.rows[0].code0 < 0 || P.rows[0].code0 >= P.V) {
            atomicOr(P.err, ERRB_BOUNDS);
            atomicExch(&P.bar[1], 1u);
        } else {
            P.codes[(size_t)c.frame * MAX_GROUPS] = P.rows[0].code0;
        }
    }
    frame_schedule<T>(c, P);
}

// ------------------------------------------------------------------ host side
template <typename T>
static size_t smem_for(int xin_bytes) {
    return align128(sizeof(FSmem<T>)) + align128((size_t)xin_bytes) + sizeof(SampSmem);
}

size_t frame_attn_scratch_bytes() { return (size_t)(2 * HD + 4 * HD + 2 * NCW * 2 + NCW * 2 * HD) * sizeof(float); }

size_t frame_smem_bytes(int dtype, int xin_bytes) {
    const size_t b = dtype == Q3_BF16 ? smem_for<bf16>(xin_bytes) : smem_for<float>(xin_bytes);
    return b <= 227 * 1024 ? b : 0;
}

cudaError_t frame_setup(int dtype, size_t smem) {
    if (dtype == Q3_BF16)
        return cudaFuncSetAttribute(frame_kernel<bf16, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return cudaFuncSetAttribute(frame_kernel<float, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t frame_occupancy(int dtype, size_t smem, int* blocks) {
    if (dtype == Q3_BF16)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, frame_kernel<bf16, 2>, NTHREADS, smem);
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, frame_kernel<float, 2>, NTHREADS, smem);
}

cudaError_t launch_frame(int dtype, const FrameParams* params_dev, int grid, size_t smem, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dtype == Q3_BF16) return cudaLaunchKernelEx(&cfg, frame_kernel<bf16, 2>, params_dev);
    return cudaLaunchKernelEx(&cfg, frame_kernel<float, 2>, params_dev);
}

}  // namespace q3
