// Persistent frame kernel: one talker step of a single row (code predictor
// 2-token prefill + 14 steps with their 15 draws, talker input assembly,
// 28-layer talker, codebook-0 selection) in ONE cooperative launch.
//
// Why: at batch 1 every projection is a GEMV that streams its weights once;
// the frame's ~3.3 GB (0.6B bf16) is bandwidth-trivial per phase (1-12 MB)
// but the phases form a ~560-long dependent chain.  Two things keep the chain
// short:
//
// * Weights do not depend on activations, so each CTA's producer warp streams
//   its slice of every upcoming projection into a shared-memory ring with bulk
//   async copies (cp.async.bulk, completion on mbarriers) as far ahead as the
//   ring allows, across phase boundaries.
// * There is no grid-wide barrier.  Every activation that crosses CTAs is a
//   64-bit word {fp32 value, epoch of the phase that wrote it}, stored with one
//   relaxed 64-bit store; a reader polls exactly the words it needs until they
//   carry the epoch it expects.  A phase therefore starts as soon as its own
//   inputs exist, and the chain pays one L2 round trip per phase instead of a
//   barrier.  Epochs are selection_index * 1024 + phase, unique per launch.
//
// Reuse of an exchange buffer is safe without a barrier because every GEMV
// phase spreads its output rows over ALL CTAs (the grid is never larger than
// the smallest output width) and every CTA reads the whole output of the
// phase before it writes anything later: a CTA that overwrites a buffer has
// transitively waited for every CTA to finish reading the previous contents.
// Each link of that chain is a store that depends on a polled value (the poll
// loop cannot exit before the load returned), so no store can become visible
// before the read it waited for; no fence is needed on this path.  Plain data
// that crosses CTAs inside a launch (attention partials) goes through the
// usual fence + counter pattern.
//
// Layout of work: a GEMV phase splits its N output rows evenly over the CTAs
// (no split-K, fixed reduction order, no atomics on values); inside a CTA each
// warp takes groups of 1-4 rows of a ring tile and keeps the rows' dot
// products in flight together.  Talker attention work items are (kv head, KV
// split): the last split of a head to finish merges the partials
// (flash-decoding combine).  Predictor attention (at most 17 positions) runs
// one item per kv head on CTA g, for every token and step, so its cache
// entries are written and read by the same CTA.  Predictor draws run on every
// CTA (same logits, same deterministic draw, same id), which removes a
// hand-off per codebook; the talker's draw runs on CTA 0.
//
// Every wait is bounded: an expired wait sets Q3's TIMEOUT error bit and the
// abort flag, which makes every other wait return; the producer then waits
// (bounded) for its own copies in flight before the CTA exits.
#include "sampler.cuh"
#include "kernels.h"
#include "frame_params.h"

#include <algorithm>
#include <type_traits>

namespace q3 {

constexpr int NCW = 8;                       // consumer warps
constexpr int NTHREADS = (NCW + 1) * 32;     // + one producer warp
// Weight ring of a kernel variant (24 KB slots): six for the tensor-core rows
// (whose row buffer of partial sums takes the room of a seventh), seven for
// the FMA rows.  Measured on config 2, more slots or wider windows of the
// tensor-core rows do not help.
template <bool TCR>
struct Ring {
    static constexpr int SLOTS = TCR ? 6 : 7;
    static constexpr int TILE = 24576;
};
constexpr int CP_VMAX = 2048;                // predictor vocabulary bound of the frame kernel
constexpr int NORM_MAX = FRAME_MAX_NORM;     // widest vector an RMSNorm prologue normalizes
constexpr int ROW_PAD = 32;                  // bytes after each bf16 weight row in the ring
constexpr int KSMAX = 8;                     // K splits of one GEMV phase (tensor-core rows)
constexpr int WT = 3;                        // ring tiles per window of tensor-core rows

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
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 2, 256;" ::: "memory"); }
// barrier of the consumer threads that also ORs a predicate over them (same result in every thread)
__device__ __forceinline__ bool consumer_sync_or(bool v) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.or.pred q, 2, 256, p;\n\t"
        "selp.s32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((int)v)
        : "memory");
    return r != 0;
}

// exchange words: relaxed gpu-scope 64-bit accesses (single-copy atomic).  No
// compiler memory clobber: what orders them is the data they carry (a store
// writes values computed from polled words), and volatile keeps every poll a
// fresh load.
__device__ __forceinline__ Word ll_ld(const Word* p) {
    Word w;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p));
    return w;
}
__device__ __forceinline__ void ll_put(Word* p, float v, unsigned ep) {
    const Word w = ((Word)ep << 32) | (Word)__float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w));
}
__device__ __forceinline__ unsigned ep_of(Word w) { return (unsigned)(w >> 32); }
__device__ __forceinline__ float val_of(Word w) { return __uint_as_float((unsigned)w); }

// data written by this CTA in an earlier phase (predictor cache) or by other
// CTAs behind a fence (attention partials): read at L2, never from L1
__device__ __forceinline__ float ldg(const float* p) { return __ldcg(p); }
__device__ __forceinline__ float ld_kv(const bf16* p) { return __bfloat162float(__ldcg(p)); }
__device__ __forceinline__ float ld_kv(const float* p) { return __ldcg(p); }

__device__ __forceinline__ bool aborted(const FrameParams& P) { return *(volatile unsigned*)&P.ctl[0] != 0u; }
__device__ __forceinline__ void raise_abort(const FrameParams& P, int bits) {
    if (bits) atomicOr(P.err, bits);
    atomicExch(&P.ctl[0], 1u);
}

// Wait on an mbarrier phase; false if the wait expired or the launch aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, unsigned parity, const FrameParams& P) {
    if (mbar_try_wait(b, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(b, parity)) {
        if (aborted(P)) return false;
        if (clock64() - t0 > P.wait_cycles) {
            raise_abort(P, ERRB_TIMEOUT);
            return false;
        }
    }
    return true;
}

// Poll N exchange words at base[first + step j] (j < N; indexes >= limit are
// skipped) until every one carries epoch e: all loads in flight together, and
// each round re-loads only the words still missing.  False if the launch
// aborted or the wait expired.  Inline on purpose: a call would make the
// caller save its live registers to local memory around every wait.
template <int N>
__device__ __forceinline__ bool ll_poll(Word (&w)[N], const Word* base, int first, int step, int limit, unsigned e,
                                        const FrameParams& P) {
    if (e == P.inject_ep) e |= 0x80000000u;   // an epoch no phase writes
#pragma unroll
    for (int j = 0; j < N; ++j) w[j] = first + step * j < limit ? ll_ld(base + first + step * j) : ((Word)e << 32);
    long long t0 = 0;
    for (unsigned it = 0;; ++it) {
        bool pend = false;
#pragma unroll
        for (int j = 0; j < N; ++j) pend |= ep_of(w[j]) != e;
        if (!pend) return true;
        if (it == 0) t0 = clock64();
        if ((it & 15u) == 15u) {
            if (aborted(P)) return false;
            if (clock64() - t0 > P.wait_cycles) {
                raise_abort(P, ERRB_TIMEOUT);
                return false;
            }
        }
#pragma unroll
        for (int j = 0; j < N; ++j)
            if (ep_of(w[j]) != e) w[j] = ll_ld(base + first + step * j);
    }
}
__device__ __forceinline__ bool ll_get(const Word* p, unsigned ep, float& v, const FrameParams& P) {
    Word w[1];
    const bool ok = ll_poll<1>(w, p, 0, 0, 1, ep, P);
    v = val_of(w[0]);
    return ok;
}
// dst[i] = src[i] (epoch ep) for this thread's i = tid, tid + 256, ... < n, four
// loads in flight; *ss accumulates v * v in that order when given.
__device__ bool ll_fetch(const Word* src, float* dst, int n, unsigned ep, float* ss, const FrameParams& P) {
    for (int i = threadIdx.x; i < n; i += 4 * 256) {
        Word w[4];
        if (!ll_poll<4>(w, src, i, 256, n, ep, P)) return false;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int k = i + j * 256;
            if (k >= n) break;
            const float v = val_of(w[j]);
            dst[k] = v;
            if (ss) *ss = fmaf(v, v, *ss);
        }
    }
    return true;
}

// ------------------------------------------------------------------ shared memory
template <typename T, bool TCR>
struct FSmem {
    static constexpr int NSLOT = Ring<TCR>::SLOTS, TILE = Ring<TCR>::TILE;
    unsigned char ring[NSLOT][TILE];
    uint64_t full[NSLOT];
    uint64_t empty[NSLOT];
    float resid[2][2][FRAME_MAX_ROWS];  // residual entries a GEMV phase updates [phase parity][vector][row]
    float pss[2][NCW][2];               // per-warp sums of squares of the RMSNorm inputs [phase parity]
    // tensor-core rows: per-split partial sums [row][gate/up][vector][split]
    float part[TCR ? FRAME_MAX_PART : 1];
    int codes[MAX_GROUPS];              // this frame's codes as drawn so far
    int flag;
    // then one region for: two input-vector buffers (one per GEMV phase
    // parity; the attention phase's scratch shares the one the next GEMV
    // phase fills) or, during a predictor draw (when no GEMV reads them), the
    // draw's scratch.  The talker's draw, the launch's last step, runs on CTA 0
    // in the drained weight ring.
};

__host__ __device__ constexpr size_t align128(size_t v) { return (v + 127) & ~(size_t)127; }
template <class S>
__device__ __forceinline__ float* xin_ptr(S& s, int buf, int xin_bytes) {
    return reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(&s) + align128(sizeof(S)) +
                                    (size_t)buf * align128((size_t)xin_bytes));
}
template <class S>
__device__ __forceinline__ SampSmemT<CP_VMAX>& samp_ptr(S& s) {
    return *reinterpret_cast<SampSmemT<CP_VMAX>*>(reinterpret_cast<unsigned char*>(&s) + align128(sizeof(S)));
}

// ------------------------------------------------------------------ the frame schedule
// Both roles walk the same schedule; the producer acts on GEMV phases and on
// the talker's attention phases only.
// prologue: NORM = rmsnorm(vector) * w; LOAD = copy the input rows; RAW = the token itself
enum class Pro { NORM, LOAD, RAW };
// where the vector comes from: the input rows (NONE) or an assembled token, whose
// residual slice this CTA also writes (NORM)
enum class Tok { NONE, CP0, CPS, TALK };
enum class Epi { STORE, ADD, BIAS, GATED };
// exchange buffers (the epoch of each one's last write is tracked per CTA)
enum Buf { BX, BCX, BQKV, BO, BACT, BLOG, BCPL, NBUF };

struct Gemv {
    const void* W;
    int N, K;
    bool gated;   // W holds [2N][K]: gate rows then up rows; output silu(g)*u
    int M;        // input vectors
    Pro pro;
    Tok tok;
    Epi epi;
    Word* src;    // NORM / LOAD: input rows; NORM with a token: its residual rows
    int src_ld, src_buf;
    const float* norm_w;
    Word* dst;
    int ld_dst, dst_buf;
    const float* bias;
    float* hout;  // NORM: also write the fp32 normed vector (talker h), this CTA's slice
    int s_idx;    // CPS / RAW: predictor step
};

__device__ __forceinline__ void split_rows(int N, int& n0, int& n1) {
    // 32-bit: N * grid stays far below 2^32 for every width of the model
    n0 = (int)(((unsigned)N * blockIdx.x) / gridDim.x);
    n1 = (int)(((unsigned)N * (blockIdx.x + 1)) / gridDim.x);
}

// Rows of a ring tile: for the tensor-core rows (TCR, bf16) rows are stored
// padded (row stride 2K + ROW_PAD bytes) so that the fragment loads of 8 rows
// hit distinct banks; otherwise rows are contiguous.
template <typename T, bool TCR>
__device__ __forceinline__ int row_stride(int K) {
    return TCR ? K * 2 + ROW_PAD : K * (int)sizeof(T);
}
template <typename T, bool TCR>
__device__ __forceinline__ int rows_per_tile(const Gemv& g) {
    const int unit = row_stride<T, TCR>(g.K) * (g.gated ? 2 : 1);
    return max(1, Ring<TCR>::TILE / unit);
}

// Cached positions [j0, j1) of talker attention split sp that the producer
// prefetches (all before the new token's position p0); false if none, or if
// they do not fit one ring slot (then the consumer reads them directly).
template <typename T, bool TCR>
__device__ __forceinline__ bool kv_prefetch_range(int p0, int S, int sp, int& j0, int& j1) {
    const int n = p0 + 1;
    const int chunk = (n + S - 1) / S;
    j0 = sp * chunk;
    j1 = min(min(n, j0 + chunk), p0);
    return j1 > j0 && (size_t)(j1 - j0) * HD * sizeof(T) * 2 <= (size_t)Ring<TCR>::TILE;
}

// ------------------------------------------------------------------ producer
template <typename T, bool TCR>
struct Producer {
    static constexpr int NSLOT = Ring<TCR>::SLOTS;
    FSmem<T, TCR>& s;
    const FrameParams& P;
    unsigned seq = 0;
    bool ok = true;
    int pos = 0;

    __device__ bool take_slot(int& slot) {
        slot = seq % NSLOT;
        const unsigned round = seq / NSLOT;
        if (round > 0 && !mbar_wait(&s.empty[slot], (round - 1) & 1, P)) { ok = false; return false; }
        ++seq;
        return true;
    }

    __device__ void gemv(const Gemv& g) {
        if (!ok) return;
        int n0, n1;
        split_rows(g.N, n0, n1);
        const int rt = rows_per_tile<T, TCR>(g);
        const size_t row_bytes = (size_t)g.K * sizeof(T);
        for (int r0 = n0; r0 < n1; r0 += rt) {
            const int r = min(rt, n1 - r0);
            int slot;
            if (!take_slot(slot)) return;
            const unsigned bytes = (unsigned)(r * row_bytes * (g.gated ? 2 : 1));
            mbar_expect_tx(&s.full[slot], bytes);
            if (TCR) {
                // one copy per row into the padded layout (gate rows, then up rows)
                const size_t rs = (size_t)row_stride<T, TCR>(g.K);
                for (int i = 0; i < r; ++i)
                    bulk_g2s(s.ring[slot] + i * rs, (const char*)g.W + (size_t)(r0 + i) * row_bytes,
                             (unsigned)row_bytes, &s.full[slot]);
                if (g.gated)
                    for (int i = 0; i < r; ++i)
                        bulk_g2s(s.ring[slot] + (r + i) * rs, (const char*)g.W + (size_t)(g.N + r0 + i) * row_bytes,
                                 (unsigned)row_bytes, &s.full[slot]);
            } else {
                bulk_g2s(s.ring[slot], (const char*)g.W + (size_t)r0 * row_bytes, (unsigned)(r * row_bytes),
                         &s.full[slot]);
                if (g.gated)
                    bulk_g2s(s.ring[slot] + r * row_bytes, (const char*)g.W + (size_t)(g.N + r0) * row_bytes,
                             (unsigned)(r * row_bytes), &s.full[slot]);
            }
        }
    }
    // Talker attention: the cached K / V of positions before the new token do
    // not depend on this step; stream each of this CTA's splits into a slot.
    __device__ void attention(int l, const PBlk& B, int M, int p0, int S, bool talker) {
        if (!ok || !talker) return;
        for (int item = blockIdx.x; item < P.nkv * S; item += gridDim.x) {
            const int g = item / S, sp = item % S;
            int j0, j1;
            if (!kv_prefetch_range<T, TCR>(p0, S, sp, j0, j1)) continue;
            int slot;
            if (!take_slot(slot)) return;
            const size_t row_bytes = (size_t)HD * sizeof(T);
            const size_t base = (((size_t)l * P.max_batch + 0) * P.nkv + g) * B.cap + j0;
            const unsigned bytes = (unsigned)((j1 - j0) * row_bytes);
            mbar_expect_tx(&s.full[slot], 2 * bytes);
            bulk_g2s(s.ring[slot], (const char*)B.Kc + base * row_bytes, bytes, &s.full[slot]);
            bulk_g2s(s.ring[slot] + bytes, (const char*)B.Vc + base * row_bytes, bytes, &s.full[slot]);
        }
    }
    __device__ void draw_cp(int) {}
    __device__ void draw_talker() {}
    __device__ void prepare_talker() {}
    __device__ int talker_pos() const { return pos; }
    __device__ bool live() const { return ok; }

    // copies issued but not yet consumed must land before the CTA exits
    __device__ void drain() {
        for (unsigned t = (seq > NSLOT ? seq - NSLOT : 0); t < seq; ++t) {
            const long long t0 = clock64();
            while (!mbar_try_wait(&s.full[t % NSLOT], (t / NSLOT) & 1))
                if (clock64() - t0 > P.wait_cycles) break;
        }
    }
};

// ------------------------------------------------------------------ GEMV helpers
__device__ __forceinline__ void lds_f32x4(uint32_t a, float& x, float& y, float& z, float& w) {
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(x), "=f"(y), "=f"(z), "=f"(w) : "r"(a));
}
// pointer through an opaque register move: reads through the result cannot be
// scheduled before the statement (a compiler barrier tied to the data)
template <typename P>
__device__ __forceinline__ P* launder(P* p) {
    unsigned long long v = reinterpret_cast<unsigned long long>(p);
    asm volatile("mov.b64 %0, %0;" : "+l"(v)::"memory");
    return reinterpret_cast<P*>(v);
}
// a shared-memory address through an opaque register move: loads from it
// cannot be scheduled before the statement
__device__ __forceinline__ uint32_t launder_u32(uint32_t v) {
    asm volatile("mov.b32 %0, %0;" : "+r"(v)::"memory");
    return v;
}
// 8-byte shared-memory load (not volatile: the compiler may batch them)
__device__ __forceinline__ uint2 lds_v2(uint32_t a) {
    uint2 r;
    asm("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(a));
    return r;
}
// D += A B for mma.m16n8k16 (bf16 in, fp32 accumulate).  a0 / a2: this lane's
// A row (lane / 4), low / high k pair; a1 / a3: the same for A row lane / 4 + 8.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// 4 consecutive elements (index multiple of 4) as fp32
__device__ __forceinline__ void load4(const bf16* p, float (&v)[4]) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    v[0] = __uint_as_float(u.x << 16); v[1] = __uint_as_float(u.x & 0xffff0000u);
    v[2] = __uint_as_float(u.y << 16); v[3] = __uint_as_float(u.y & 0xffff0000u);
}
__device__ __forceinline__ void load4(const float* p, float (&v)[4]) {
    const float4 f = *reinterpret_cast<const float4*>(p);
    v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
}
// 4 consecutive elements at shared address a as fp32
__device__ __forceinline__ void lds4(uint32_t a, float (&v)[4], float) { lds_f32x4(a, v[0], v[1], v[2], v[3]); }
__device__ __forceinline__ void lds4(uint32_t a, float4& v) { lds_f32x4(a, v.x, v.y, v.z, v.w); }
__device__ __forceinline__ void lds4(uint32_t a, float (&v)[4], bf16) {
    uint32_t x, y;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(x), "=r"(y) : "r"(a));
    v[0] = __uint_as_float(x << 16); v[1] = __uint_as_float(x & 0xffff0000u);
    v[2] = __uint_as_float(y << 16); v[3] = __uint_as_float(y & 0xffff0000u);
}

// Sums of V = 2^n values over the warp with V - 1 + (5 - n) shuffles: each
// halving step keeps one half of the values in each half of the lanes.  Lane l
// ends with the full sum of value j(l) = sum_s bit(l, 4 - s) * V / 2^(s + 1)
// (s = 0 .. n-1); lanes that differ only in the low 5 - n bits hold the same value.
template <int N, int OFF, int V>
__device__ __forceinline__ void split_step(float (&v)[V], int lane) {
    if constexpr (OFF >= 1) {
        if constexpr (N > 1) {
            const bool upper = (lane & OFF) != 0;
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                const float send = upper ? v[i] : v[i + N / 2];
                const float keep = upper ? v[i + N / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
            }
            split_step<N / 2, OFF / 2, V>(v, lane);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], OFF);
            split_step<1, OFF / 2, V>(v, lane);
        }
    }
}
template <int V>
__device__ __forceinline__ float warp_sum_split(float (&v)[V], int lane) {
    static_assert(V >= 1 && V <= 32 && (V & (V - 1)) == 0, "V must be a power of two");
    split_step<V, 16, V>(v, lane);
    return v[0];
}
// the value index lane l holds after warp_sum_split<V>
template <int V>
__device__ __forceinline__ int split_index(int lane) {
    int j = 0, half = V / 2, bit = 16;
#pragma unroll
    for (int st = 0; st < 5; ++st) {
        if (half >= 1) {
            if (lane & bit) j += half;
            half >>= 1;
            bit >>= 1;
        }
    }
    return j;
}

// ------------------------------------------------------------------ consumer
template <typename T, int GQ, bool TCR>
struct Consumer {
    static constexpr int NSLOT = Ring<TCR>::SLOTS, TILE = Ring<TCR>::TILE;
    FSmem<T, TCR>& s;
    const FrameParams& P;
    unsigned seq = 0;        // ring slots consumed
    unsigned base = 0;       // epoch of this launch's phase 0
    unsigned ph = 0;         // phases walked
    unsigned gph = 0;        // GEMV phases walked (picks the partials buffer)
    unsigned ep[NBUF] = {};  // epoch of the last write of each exchange buffer
    int frame = 0;           // frame completed by this step
    int pos = 0;             // talker position of the new token
    bool ok = true;          // uniform over the CTA's consumer threads (changes in settle only)
    bool failed = false;     // a wait of this thread failed (reported at the next settle)

    // input-vector buffer of the next GEMV phase (also the attention scratch)
    __device__ float* xin_next() { return xin_ptr(s, (int)(gph & 1), P.xin_bytes); }
    __device__ unsigned next_phase() { return base + ph++; }

    // Every thread reports whether its waits succeeded (and any wait that failed
    // earlier in this thread); all get the same answer: false if any failed.
    __device__ bool settle(bool good) {
        if (!good) failed = true;
        if (consumer_sync_or(failed)) ok = false;
        return ok;
    }

    __device__ bool live() const { return ok; }

    // value i (talker width) of input vector m of an assembled-token phase
    __device__ __forceinline__ float token_value(Tok tok, int s_idx, int m, int i) {
        const int H = P.H;
        if (tok == Tok::TALK) return talker_input(i);
        if (tok == Tok::CP0) {
            if (m == 0) return ldg(P.h + i);
            return to_f(((const T*)P.codec_emb)[(size_t)s.codes[0] * H + i]);
        }
        return to_f(((const T*)P.cp_emb)[((size_t)(s_idx - 1) * P.cpV + s.codes[s_idx]) * H + i]);
    }

    // talker input: codec_emb(code0) + sum_q table[q-1](code_q) + text row
    const float* tk_text = nullptr;
    __device__ void prepare_talker() {
        if (!ok) return;
        const RowState& rs = P.rows[0];
        tk_text = frame < rs.n_text ? P.text + (size_t)(rs.text_off + frame) * P.H : P.pad;
    }
    __device__ int talker_pos() const { return pos; }
    __device__ float talker_input(int i) {
        const int H = P.H;
        float acc = to_f(((const T*)P.codec_emb)[(size_t)s.codes[0] * H + i]);
        for (int q = 1; q < P.G; ++q)
            acc += to_f(((const T*)P.cp_emb)[((size_t)(q - 1) * P.cpV + s.codes[q]) * H + i]);
        return acc + tk_text[i];
    }

    // The rows of a GEMV phase on the tensor cores (bf16 weights).  Each
    // mma.m16n8k16 multiplies 16 weight rows (A) with the input vectors (B:
    // column 2m is vector m's bf16 high part, column 2m + 1 its low part) over
    // 16 elements of K, so one instruction gives both parts of 16 dot products.
    // The K order inside a 16-element step is permuted so that a lane's A and B
    // fragments are 4 consecutive elements (one 8-byte load each): MMA k pairs
    // (2q, 2q+1) and (2q+8, 2q+9) are elements 4q..4q+3.
    // The phase's tiles are taken WT at a time (all resident); a window's rows
    // form 16-row blocks (across tiles), and (block, K split) units are dealt to
    // the warps; their partial sums meet in shared memory, and after the
    // phase's second barrier one thread per output adds the splits in order.
    template <int M, bool GATED>
    __device__ void rows_tc(const Gemv& g, unsigned cur, int buf, const float (&rm)[2], int n0, int nrows) {
        constexpr int H2 = GATED ? 2 : 1;
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int K = g.K, nks = K >> 4;
        const int rt = rows_per_tile<T, TCR>(g);
        const size_t rs = (size_t)row_stride<T, TCR>(K);
        const int ntiles = (nrows + rt - 1) / rt;
        const int nbw = (min(WT * rt, nrows) + 15) >> 4;   // blocks of a full window
        const int ks = max(1, min(KSMAX, NCW / nbw));
        const int gq = lane >> 2, q = lane & 3;
        // B fragment: this lane supplies column gq (vector gq / 2, high part if
        // gq is even); columns from 2M on are zero
        const bool xcol = gq < 2 * M;
        // the vector was stored before the phase's barrier; its address is taken after it
        const uint32_t xa = launder_u32(smem_u32(xin_ptr(s, buf, P.xin_bytes))) +
                            (uint32_t)(((gq & 1) * M + min(gq >> 1, M - 1)) * K * 2 + q * 8);
        float* part = s.part;
        bool good = true;
        for (int w0 = 0; w0 < ntiles; w0 += WT) {
            const int wt = min(WT, ntiles - w0);
            const unsigned seqw = seq;
            for (int t = 0; t < wt; ++t) {
                const unsigned sq = seqw + t;
                good = good && mbar_wait(&s.full[sq % NSLOT], (sq / NSLOT) & 1, P);
            }
            seq += wt;
            // ring addresses taken after the waits
            const uint32_t ring = launder_u32(smem_u32(&s.ring[0][0]));
            const int row_w0 = w0 * rt;
            const int rw = min(wt * rt, nrows - row_w0);
            const int nb = (rw + 15) >> 4;
            for (int u = warp; good && u < nb * ks; u += NCW) {
                const int b = u / ks, kq = u - b * ks;
                const int k0 = nks * kq / ks, k1 = nks * (kq + 1) / ks;
                // this lane's A rows of the block: gq and gq + 8 (clamped into the window)
                uint32_t wa[2], ua[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int j = min(b * 16 + gq + 8 * h, rw - 1);
                    const int t = j / rt, i = j - t * rt;
                    const int rtile = min(rt, nrows - row_w0 - t * rt);
                    const uint32_t tb = ring + (uint32_t)(((seqw + t) % NSLOT) * TILE);
                    wa[h] = tb + (uint32_t)(i * rs + q * 8);
                    ua[h] = tb + (uint32_t)((rtile + i) * rs + q * 8);
                }
                float d[4][H2][4];
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int h = 0; h < H2; ++h)
#pragma unroll
                        for (int e = 0; e < 4; ++e) d[c][h][e] = 0.f;
                // four K steps at a time, every load of the four issued before their MMAs
                int k = k0;
                for (; k + 4 <= k1; k += 4) {
                    uint2 xv[4], w0[4], w1[4], u0[GATED ? 4 : 1], u1[GATED ? 4 : 1];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t o = (uint32_t)(k + c) * 32u;
                        xv[c] = make_uint2(0u, 0u);
                        if (xcol) xv[c] = lds_v2(xa + o);
                        w0[c] = lds_v2(wa[0] + o);
                        w1[c] = lds_v2(wa[1] + o);
                        if constexpr (GATED) {
                            u0[c] = lds_v2(ua[0] + o);
                            u1[c] = lds_v2(ua[1] + o);
                        }
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        mma_bf16(d[c][0], w0[c].x, w1[c].x, w0[c].y, w1[c].y, xv[c].x, xv[c].y);
                        if constexpr (GATED)
                            mma_bf16(d[c][H2 - 1], u0[c].x, u1[c].x, u0[c].y, u1[c].y, xv[c].x, xv[c].y);
                    }
                }
                for (; k < k1; ++k) {
                    const uint32_t o = (uint32_t)k * 32u;
                    uint2 xv = make_uint2(0u, 0u);
                    if (xcol) xv = lds_v2(xa + o);
                    const uint2 a0 = lds_v2(wa[0] + o), a1 = lds_v2(wa[1] + o);
                    mma_bf16(d[0][0], a0.x, a1.x, a0.y, a1.y, xv.x, xv.y);
                    if constexpr (GATED) {
                        const uint2 g0 = lds_v2(ua[0] + o), g1 = lds_v2(ua[1] + o);
                        mma_bf16(d[0][H2 - 1], g0.x, g1.x, g0.y, g1.y, xv.x, xv.y);
                    }
                }
                // lane 4 r + q (q < M) holds vector q's high and low sums of
                // rows r (d[0], d[1]) and r + 8 (d[2], d[3]) of the block
                if (q < M) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int jr = b * 16 + gq + 8 * e;
                        if (jr < rw) {
                            const int prow = row_w0 + jr;
#pragma unroll
                            for (int h = 0; h < H2; ++h)
                                part[((prow * H2 + h) * M + q) * KSMAX + kq] =
                                    ((d[0][h][2 * e] + d[0][h][2 * e + 1]) + (d[1][h][2 * e] + d[1][h][2 * e + 1])) +
                                    ((d[2][h][2 * e] + d[2][h][2 * e + 1]) + (d[3][h][2 * e] + d[3][h][2 * e + 1]));
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                for (int t = 0; t < wt; ++t) mbar_arrive(&s.empty[(seqw + t) % NSLOT]);
        }
        if (!good) failed = true;
        // every partial is in place (and a failed wait is known to every warp)
        if (!settle(good)) return;
        for (int o = threadIdx.x; o < nrows * M; o += 256) {
            const int row = o / M, m = o - row * M, n = n0 + row;
            float a = 0.f, up = 0.f;
            for (int kq = 0; kq < ks; ++kq) {
                a += part[((row * H2) * M + m) * KSMAX + kq];
                if (GATED) up += part[((row * H2 + 1) * M + m) * KSMAX + kq];
            }
            const float r_m = m == 0 ? rm[0] : rm[1];
            a *= r_m;
            float out;
            if (GATED) out = a / (1.0f + expf(-a)) * (up * r_m);
            else if (g.epi == Epi::ADD) out = s.resid[buf][m][row] + a;
            else if (g.epi == Epi::BIAS) out = a + g.bias[n];
            else out = a;
            ll_put(g.dst + (size_t)m * g.ld_dst + n, out, cur);
        }
    }

    // One GEMV phase.  Prologue: each thread fetches input elements i = tid,
    // tid + 256, ... (polled exchange words or an assembled token), forms
    // x (.) w for RMSNorm phases and stores it in this phase's shared buffer,
    // and sums x^2; ADD phases also fetch the residual entries they update.  One
    // barrier.  Then each warp takes groups of RG rows of the ring tiles,
    // round-robin over the phase, keeps their dot products with the whole
    // vector in flight, reduces them over the lanes together, and the lanes
    // holding the sums write the outputs.  RMSNorm is applied as the scalar it
    // is: W (x r (.) w) = r W (x (.) w), with r from the warps' sums of squares.
    template <int RG, int M, bool GATED>
    __device__ void gemv_run(const Gemv& g, unsigned cur) {
        constexpr int H2 = GATED ? 2 : 1;
        constexpr int V = RG * M * H2;
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
        const int K = g.K;
        const bool norm = g.pro == Pro::NORM;
        const bool tok = g.tok != Tok::NONE;
        int n0, n1;
        split_rows(g.N, n0, n1);
        const int nrows = n1 - n0;
        const int buf = gph & 1;
        float* xs = xin_ptr(s, buf, P.xin_bytes);
        ++gph;
        bool good = true;
        // the input vectors in this phase's buffer: fp32 [M][K] for the FMA rows,
        // bf16 high and low parts [M][K] each for the tensor-core rows
        auto put_x = [&](int m, int i, float v) {
            if constexpr (TCR) {
                bf16* xh = reinterpret_cast<bf16*>(xs);
                const bf16 h = __float2bfloat16_rn(v);
                xh[m * K + i] = h;
                xh[(M + m) * K + i] = __float2bfloat16_rn(v - __bfloat162float(h));
            } else {
                xs[m * K + i] = v;
            }
        };

        // this thread's RMSNorm weights (K <= NORM_MAX), fetched before any wait
        float nw[NORM_MAX / 256];
        if (norm) {
#pragma unroll
            for (int j = 0; j < NORM_MAX / 256; ++j) nw[j] = tid + 256 * j < K ? g.norm_w[tid + 256 * j] : 0.f;
        }
        // residual entries this CTA updates
        if (g.epi == Epi::ADD && tid < nrows * M) {
            float v = 0.f;
            good = ll_get(g.dst + (size_t)(tid % M) * g.ld_dst + n0 + tid / M, ep[g.dst_buf], v, P);
            s.resid[buf][tid % M][tid / M] = v;
        }
        float ssq[2] = {0.f, 0.f};
        constexpr int NJ = NORM_MAX / 256;
        if (!tok && norm) {
            // K <= NORM_MAX: all of this thread's words in flight at once
            const unsigned e = ep[g.src_buf];
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const Word* src = g.src + (size_t)m * g.src_ld;
                Word w[NJ];
                good = ll_poll<NJ>(w, src, tid, 256, K, e, P) && good;
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    const int i = tid + 256 * j;
                    if (i < K) {
                        const float v = val_of(w[j]);
                        ssq[m] = fmaf(v, v, ssq[m]);
                        put_x(m, i, v * nw[j]);
                    }
                }
            }
        } else if (!tok) {
            // up to 12 words per thread in flight at once: one L2 round trip
            // for inputs up to 3072 wide (attention output, SiLU(g)*u)
            const unsigned e = ep[g.src_buf];
            constexpr int NW = 12;
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const Word* src = g.src + (size_t)m * g.src_ld;
                for (int i0 = tid; i0 < K && good; i0 += NW * 256) {
                    Word w[NW];
                    good = ll_poll<NW>(w, src, i0, 256, K, e, P);
#pragma unroll
                    for (int q = 0; q < NW; ++q)
                        if (i0 + q * 256 < K) put_x(m, i0 + q * 256, val_of(w[q]));
                }
            }
        } else {
            // an assembled token (K = talker width <= NORM_MAX): every CTA builds
            // the whole vector; with NORM it also publishes the CTA's slice of
            // the residual rows
            int r0 = 0, r1 = 0;
            if (norm) split_rows(K, r0, r1);
#pragma unroll
            for (int m = 0; m < M; ++m) {
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    const int i = tid + 256 * j;
                    if (i < K) {
                        float v = token_value(g.tok, g.s_idx, m, i);
                        if (norm) {
                            if (i >= r0 && i < r1) ll_put(g.src + (size_t)m * g.src_ld + i, v, cur);
                            ssq[m] = fmaf(v, v, ssq[m]);
                            v *= nw[j];
                        }
                        put_x(m, i, v);
                    }
                }
            }
        }
        if (norm) {
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const float q = warp_sum(ssq[m]);
                if (lane == 0) s.pss[buf][warp][m] = q;
            }
        }
        // the phase's one barrier (also makes a failed wait known to every thread)
        if (!settle(good)) return;
        float rm[2] = {1.f, 1.f};
        if (norm) {
#pragma unroll
            for (int m = 0; m < M; ++m) {
                float q = 0.f;
#pragma unroll
                for (int w = 0; w < NCW; ++w) q += s.pss[buf][w][m];
                rm[m] = 1.0f / sqrtf(q / (float)K + P.eps);
            }
        }
        if (g.hout) {
            // this CTA's slice of the normed vector (the talker's h, read by the next step)
            int h0, h1;
            split_rows(K, h0, h1);
            for (int i = h0 + tid; i < h1; i += 256) {
                float xv;
                if constexpr (TCR) {
                    const bf16* xh = reinterpret_cast<const bf16*>(xs);
                    xv = __bfloat162float(xh[i]) + __bfloat162float(xh[M * K + i]);
                } else {
                    xv = xs[i];
                }
                g.hout[i] = xv * rm[0];
            }
        }
        if constexpr (TCR) {
            rows_tc<M, GATED>(g, cur, buf, rm, n0, nrows);
            if (tok && norm) ep[g.src_buf] = cur;
            return;
        }

        // the rows, as they arrive.  A lane covers elements k + 4 l .. k + 4 l + 3
        // and k + 128 + 4 l .. (l = lane) of every 256-element block k: its
        // shared-memory reads of the vector and of a row are contiguous across
        // the warp (no bank conflicts), and the vector is read once per group.
        const int rt = rows_per_tile<T, TCR>(g);
        const int gpt = (rt + RG - 1) / RG;   // row groups of a full tile
        const size_t row_bytes = (size_t)K * sizeof(T);
        const int jv = split_index<V>(lane);
        const int jr = jv / (M * H2), jm = (jv / H2) % M;
        constexpr int NB = V == 16 ? 4 : (V == 8 ? 3 : (V == 4 ? 2 : (V == 2 ? 1 : 0)));
        // the lane that writes value jv: lowest lane of its duplicates, gate half for gated
        const bool writer = (lane & ((1 << (5 - NB)) - 1)) == 0 && (!GATED || (jv % H2) == 0);
        int t = 0;
        for (int r0 = n0; r0 < n1; r0 += rt, ++t) {
            const int r = min(rt, n1 - r0);
            const int slot = seq % NSLOT;
            const unsigned round = seq / NSLOT;
            ++seq;
            if (!mbar_wait(&s.full[slot], round & 1, P)) { failed = true; return; }
            // the tile's address passes through an opaque step after the wait, so
            // no read of it can be scheduled before the data has landed
            const unsigned char* tile = launder(s.ring[slot]);
            const int ng = (r + RG - 1) / RG;
            for (int q = (warp - (t * gpt) % NCW + NCW) % NCW; q < ng; q += NCW) {
                const int i0 = q * RG;
                const int nr = min(RG, r - i0);
                const T* wrow[H2][RG];
#pragma unroll
                for (int h = 0; h < H2; ++h)
#pragma unroll
                    for (int rr = 0; rr < RG; ++rr)
                        wrow[h][rr] = reinterpret_cast<const T*>(tile + (size_t)(h * r + i0 + min(rr, nr - 1)) * row_bytes);
                // U accumulator sets (fewer for wide groups: 9 warps leave 168
                // registers a thread): blocks of 128 elements, lane l on 4 l .. 4 l + 3
                constexpr int U = H2 * RG * M <= 4 ? 4 : (H2 * RG * M <= 8 ? 2 : 1);
                float acc[U][H2][RG][M];
#pragma unroll
                for (int a = 0; a < U; ++a)
#pragma unroll
                    for (int h = 0; h < H2; ++h)
#pragma unroll
                        for (int rr = 0; rr < RG; ++rr)
#pragma unroll
                            for (int m = 0; m < M; ++m) acc[a][h][rr][m] = 0.f;
                auto block = [&](int k, float (&A)[H2][RG][M]) {
                    float4 xv[M];
#pragma unroll
                    for (int m = 0; m < M; ++m) xv[m] = *reinterpret_cast<const float4*>(xs + m * K + k);
#pragma unroll
                    for (int h = 0; h < H2; ++h)
#pragma unroll
                        for (int rr = 0; rr < RG; ++rr) {
                            float wv[4];
                            load4(wrow[h][rr] + k, wv);
#pragma unroll
                            for (int m = 0; m < M; ++m) {
                                float& c = A[h][rr][m];
                                c = fmaf(wv[0], xv[m].x, c);
                                c = fmaf(wv[1], xv[m].y, c);
                                c = fmaf(wv[2], xv[m].z, c);
                                c = fmaf(wv[3], xv[m].w, c);
                            }
                        }
                };
                int kb = 0;
                for (; kb + 128 * U <= K; kb += 128 * U) {
#pragma unroll
                    for (int a = 0; a < U; ++a) block(kb + 128 * a + lane * 4, acc[a]);
                }
                for (; kb < K; kb += 128)
                    if (kb + lane * 4 < K) block(kb + lane * 4, acc[0]);
                // value index (rr * M + m) * H2 + h
                float v[V];
#pragma unroll
                for (int h = 0; h < H2; ++h)
#pragma unroll
                    for (int rr = 0; rr < RG; ++rr)
#pragma unroll
                        for (int m = 0; m < M; ++m) {
                            float sacc = acc[0][h][rr][m];
#pragma unroll
                            for (int a = 1; a < U; ++a) sacc += acc[a][h][rr][m];
                            v[(rr * M + m) * H2 + h] = sacc;
                        }
                const float sum = warp_sum_split<V>(v, lane);
                // gated: the up sum of the same output sits in the next value index
                const float up = GATED ? __shfl_down_sync(0xffffffffu, sum, 1 << (5 - NB)) : 0.f;
                if (writer && jr < nr) {
                    const int n = r0 + i0 + jr;
                    const float rr_m = jm == 0 ? rm[0] : rm[1];
                    const float a = sum * rr_m;
                    float o;
                    if (GATED) {
                        const float u = up * rr_m;
                        o = a / (1.0f + expf(-a)) * u;
                    } else if (g.epi == Epi::ADD) {
                        o = s.resid[buf][jm][n - n0] + a;
                    } else if (g.epi == Epi::BIAS) {
                        o = a + g.bias[n];
                    } else {
                        o = a;
                    }
                    ll_put(g.dst + (size_t)jm * g.ld_dst + n, o, cur);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.empty[slot]);
        }
        if (tok && norm) ep[g.src_buf] = cur;
    }

    template <int RG>
    __device__ void gemv_rg(const Gemv& g, unsigned cur) {
        if (g.gated) {
            if (g.M == 1) gemv_run<RG, 1, true>(g, cur); else gemv_run<RG, 2, true>(g, cur);
        } else {
            if (g.M == 1) gemv_run<RG, 1, false>(g, cur); else gemv_run<RG, 2, false>(g, cur);
        }
    }

    __device__ void gemv(const Gemv& g) {
        const unsigned cur = next_phase();
        if (!ok) return;
        int n0, n1;
        split_rows(g.N, n0, n1);
        const int nrows = n1 - n0, rt = rows_per_tile<T, TCR>(g);
        int rg = nrows >= 3 * NCW ? 4 : (nrows >= 3 * NCW / 2 ? 2 : 1);
        while (rg > rt) rg >>= 1;
        if (TCR) gemv_rg<1>(g, cur);   // tensor-core rows; no row groups
        else if (rg == 4) gemv_rg<4>(g, cur);
        else if (rg == 2) gemv_rg<2>(g, cur);
        else gemv_rg<1>(g, cur);
        ep[g.dst_buf] = cur;
    }

    // ---------------- attention for M new tokens at positions p0.. of a layer
    // smem use (the scratch region): q [M][GQ][HD], new
    // k / v [M][HD] each (rounded as cached), per-warp softmax state.
    __device__ void attention(int l, const PBlk& B, int M, int p0, int S, bool talker) {
        const unsigned cur = next_phase();
        if (!ok) return;
        const int nq = P.nq, nkv = P.nkv;
        const int nqkv = (nq + 2 * nkv) * HD;
        const int items = talker ? nkv * S : nkv;
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        float* sq = xin_next();               // [2][GQ][HD]
        float* sk = sq + 2 * GQ * HD;         // [2][HD]
        float* sv = sk + 2 * HD;              // [2][HD]
        float* sm_m = sv + 2 * HD;            // [NCW][GQ]
        float* sm_l = sm_m + NCW * GQ;        // [NCW][GQ]
        float* sacc = sm_l + NCW * GQ;        // [NCW][GQ][HD]
        const unsigned eq = ep[BQKV];
        for (int item = blockIdx.x; item < items; item += gridDim.x) {
            const int g = talker ? item / S : item;
            const int sp = talker ? item % S : 0;
            // q heads of group g and the new k / v of tokens 0..M-1: QK-norm + RoPE
            bool good = true;
            constexpr int per = GQ + 2;
            for (int t = warp; t < M * per; t += NCW) {
                const int m = t / per, u = t % per;
                const Word* src;
                float* dst;
                const float* wn = nullptr;
                bool rope = true, kv = true;
                if (u < GQ) {
                    src = P.qkv + (size_t)m * nqkv + (size_t)(g * GQ + u) * HD;
                    dst = sq + (m * GQ + u) * HD; wn = B.q_norm + (size_t)l * HD; kv = false;
                } else if (u == GQ) {
                    src = P.qkv + (size_t)m * nqkv + (size_t)(nq + g) * HD;
                    dst = sk + m * HD; wn = B.k_norm + (size_t)l * HD;
                } else {
                    src = P.qkv + (size_t)m * nqkv + (size_t)(nq + nkv + g) * HD;
                    dst = sv + m * HD; rope = false;
                }
                // norm weights and rotation first: they do not depend on the wait
                float wnv[4] = {1.f, 1.f, 1.f, 1.f};
                float2 c0 = make_float2(1.f, 0.f), c1 = make_float2(1.f, 0.f);
                if (rope) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) wnv[i] = wn[lane + 32 * i];
                    const int tp = p0 + m;
                    c0 = P.rope[(size_t)tp * (HD / 2) + lane];
                    c1 = P.rope[(size_t)tp * (HD / 2) + lane + 32];
                }
                Word wq[4];
                good = ll_poll<4>(wq, src, lane, 32, HD, eq, P) && good;
                float e[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) e[i] = val_of(wq[i]);
                if (rope) {
                    const float ss = warp_sum(e[0] * e[0] + e[1] * e[1] + e[2] * e[2] + e[3] * e[3]);
                    const float r = 1.0f / sqrtf(ss / (float)HD + P.eps);
#pragma unroll
                    for (int i = 0; i < 4; ++i) e[i] = e[i] * r * wnv[i];
                    float a = e[0], b = e[2];
                    e[0] = a * c0.x - b * c0.y; e[2] = b * c0.x + a * c0.y;
                    a = e[1]; b = e[3];
                    e[1] = a * c1.x - b * c1.y; e[3] = b * c1.x + a * c1.y;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[lane + 32 * i] = kv ? to_f(from_f<T>(e[i])) : e[i];
            }
            if (!settle(good)) return;
            // cache [L][max_batch][nkv][cap][HD], row 0
            T* Kg = (T*)B.Kc + (((size_t)l * P.max_batch + 0) * nkv + g) * B.cap * HD;
            T* Vg = (T*)B.Vc + (((size_t)l * P.max_batch + 0) * nkv + g) * B.cap * HD;
            for (int m = 0; m < M; ++m) {
                const int pos = p0 + m;
                const int n = pos + 1;
                const int chunk = (n + S - 1) / S;
                const int j0 = sp * chunk, j1 = min(n, j0 + chunk);
                // the split holding the token's own position appends its k / v
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
                bool ring_ok = true;
                if (talker && kv_prefetch_range<T, TCR>(p0, S, sp, pj0, pj1)) {
                    slot = seq % NSLOT;
                    const unsigned round = seq / NSLOT;
                    ++seq;
                    ring_ok = mbar_wait(&s.full[slot], round & 1, P);
                    kring = (const T*)s.ring[slot];
                    vring = kring + (size_t)(pj1 - pj0) * HD;
                }
                // online softmax over positions j0..j1-1, one position per warp step
                float mx[GQ], lsum[GQ], acc[GQ][4];
                const float* q = sq + m * GQ * HD;
#pragma unroll
                for (int hh = 0; hh < GQ; ++hh) {
                    mx[hh] = -INFINITY; lsum[hh] = 0.f;
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[hh][i] = 0.f;
                }
                const float scale = 0.08838834764831845f;
                for (int j = j0 + warp; j < j1 && ring_ok; j += NCW) {
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
                        for (int i = 0; i < 4; ++i) d = fmaf(q[hh * HD + lane + 32 * i], kk[i], d);
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
                if (!settle(ring_ok)) return;
                Word* o = P.o + (size_t)m * nq * HD + (size_t)g * GQ * HD;
                if (S == 1) {
                    // one split: merge the warps straight into the output words
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
                        ll_put(o + idx, a / ls, cur);
                    }
                    consumer_sync();
                    continue;
                }
                // this split's partial
                float* part = P.part + (((size_t)g * S + sp) * GQ) * (HD + 2);
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
                // the last split of this head group to finish merges all splits
                consumer_sync();
                if (threadIdx.x == 0) {
                    __threadfence();
                    const unsigned old = atomicAdd(&P.ctl[8 + g], 1u);
                    const int last = old == (unsigned)S - 1;
                    if (last) atomicExch(&P.ctl[8 + g], 0u);
                    s.flag = last;
                }
                consumer_sync();
                if (s.flag) {
                    __threadfence();
                    const float* pb = P.part + ((size_t)g * S) * GQ * (HD + 2);
                    for (int idx = threadIdx.x; idx < GQ * HD; idx += 256) {
                        const int hh = idx / HD, d = idx % HD;
                        float ma = -INFINITY;
                        for (int qs = 0; qs < S; ++qs) ma = fmaxf(ma, ldg(pb + ((size_t)qs * GQ + hh) * (HD + 2) + HD));
                        float num = 0.f, den = 0.f;
                        for (int qs = 0; qs < S; ++qs) {
                            const float* pq = pb + ((size_t)qs * GQ + hh) * (HD + 2);
                            const float mq = ldg(pq + HD);
                            const float c = (mq == -INFINITY) ? 0.f : expf(mq - ma);
                            num += ldg(pq + d) * c;
                            den += ldg(pq + HD + 1) * c;
                        }
                        ll_put(o + idx, num / den, cur);
                    }
                }
                consumer_sync();
            }
        }
        ep[BO] = cur;
    }

    // ---------------- draws
    // Predictor draw s on every CTA: the same logits and the same deterministic
    // draw give every CTA the same id; CTA 0 records it.
    __device__ void draw_cp(int sidx) {
        next_phase();
        if (!ok) return;
        // the draw's scratch overlays the input buffers: every warp must be done
        // with the head's rows first
        consumer_sync();
        auto& sm = samp_ptr(s);
        if (!settle(ll_fetch(P.cpl, sm.l, P.cpV, ep[BCPL], nullptr, P))) return;
        const q3tts_sampling p = P.P[0];
        if (blockIdx.x == 0 && P.cap_c && P.cap_slot[0] >= 0 && frame < P.cap_T) {
            float* dst = P.cap_c + (((size_t)P.cap_slot[0] * P.cap_T + frame) * (P.G - 1) + sidx) * P.cpV;
            for (int i = threadIdx.x; i < P.cpV; i += 256) dst[i] = sm.l[i];
        }
        const DrawCfg d{p.cp_do_sample, p.cp_temperature, p.cp_top_k, p.cp_top_p};
        const int id = sample_row(sm, nullptr, P.cpV, d, false, 1.0f, nullptr, nullptr, 0, 0, -1, 0, 0, p.seed, 0u,
                                  (uint32_t)frame, (uint32_t)(sidx + 1));
        if (id < 0) {
            if (threadIdx.x == 0) {
                if (blockIdx.x == 0) {
                    RowState& rs = P.rows[0];
                    rs.finished = 1;
                    rs.reason = Q3_FINISHED_ERROR;
                    rs.frames = frame;
                }
                raise_abort(P, ERRB_NAN);
            }
            ok = false;
            return;
        }
        if (threadIdx.x == 0) {
            s.codes[sidx + 1] = id;
            if (blockIdx.x == 0) P.codes[(size_t)frame * MAX_GROUPS + sidx + 1] = id;
        }
        consumer_sync();
    }

    __device__ void draw_talker() {
        next_phase();
        if (!ok || blockIdx.x != 0) return;
        // the launch's last step: every weight tile has been consumed, so the
        // draw's scratch (the full vocabulary) can live in the drained ring
        static_assert(sizeof(SampSmem) <= sizeof(s.ring), "talker draw scratch must fit the ring");
        consumer_sync();
        SampSmem& sm = *reinterpret_cast<SampSmem*>(&s.ring[0][0]);
        if (!settle(ll_fetch(P.logits, sm.l, P.V, ep[BLOG], nullptr, P))) return;
        RowState& rs = P.rows[0];
        const q3tts_sampling p = P.P[0];
        const int k = frame + 1;
        if (P.cap_t && P.cap_slot[0] >= 0 && k <= P.cap_T) {
            float* dst = P.cap_t + ((size_t)P.cap_slot[0] * (P.cap_T + 1) + k) * P.V;
            for (int i = threadIdx.x; i < P.V; i += 256) dst[i] = sm.l[i];
        }
        const DrawCfg d{p.do_sample, p.temperature, p.top_k, p.top_p};
        int id = sample_row(sm, nullptr, P.V, d, true, p.repetition_penalty, rs.seen, nullptr, k, p.min_new_tokens,
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
// The step is a flat list of phases walked by one loop, so that each kind of
// phase has exactly one call site: one copy of its code, which stays in the
// instruction cache from one use to the next (a call site per layer phase
// would inline a separate copy of the same GEMV code for each).
enum class Ph { PROJ, QKV, ATTN, O, GU, DOWN, HEAD, DRAW_CP, PREP_T, DRAW_T };

struct PhaseAt {
    Ph kind;
    int s;         // predictor pass (codebook s + 1 is drawn at its end)
    int l;         // layer
    bool talker;
};

// phase i of the step: predictor passes s = 0..G-2 ([projection], 5 phases per
// layer, head, draw), then the talker (prepare, 5 phases per layer, head, draw)
__device__ __forceinline__ PhaseAt phase_at(int i, const FrameParams& P) {
    const int proj = P.H != P.Hc ? 1 : 0;
    const int per_pass = proj + 5 * P.c.L + 2;
    const int n_pred = (P.G - 1) * per_pass;
    PhaseAt a{Ph::PREP_T, 0, 0, false};
    int j;
    int L;
    if (i < n_pred) {
        a.s = i / per_pass;
        j = i - a.s * per_pass;
        if (proj && j == 0) { a.kind = Ph::PROJ; return a; }
        j -= proj;
        L = P.c.L;
    } else {
        a.talker = true;
        j = i - n_pred;
        if (j == 0) return a;   // PREP_T
        j -= 1;
        L = P.t.L;
    }
    if (j < 5 * L) {
        a.l = j / 5;
        a.kind = (Ph)((int)Ph::QKV + j % 5);
    } else {
        a.kind = j == 5 * L ? Ph::HEAD : (a.talker ? Ph::DRAW_T : Ph::DRAW_CP);
    }
    return a;
}

__device__ __forceinline__ int phase_count(const FrameParams& P) {
    const int proj = P.H != P.Hc ? 1 : 0;
    return (P.G - 1) * (proj + 5 * P.c.L + 2) + 1 + 5 * P.t.L + 2;
}

// the GEMV of a projection, layer or head phase
template <typename T>
__device__ __forceinline__ Gemv phase_gemv(const PhaseAt& a, const FrameParams& P) {
    const size_t e = sizeof(T);
    const PBlk& B = a.talker ? P.t : P.c;
    const int nq = P.nq, nkv = P.nkv, H = B.H, F = B.F, l = a.l;
    const int nqkv = (nq + 2 * nkv) * HD;
    const int M = (!a.talker && a.s == 0) ? 2 : 1;
    Word* x = a.talker ? P.x : P.cx;
    const int xb = a.talker ? BX : BCX;
    // the token a pass starts from: assembled by the first GEMV that reads it
    const Tok first_tok = a.talker ? Tok::TALK : (a.s == 0 ? Tok::CP0 : Tok::CPS);
    const bool proj = P.H != P.Hc;
    Gemv g{};
    g.M = M;
    g.s_idx = a.talker ? 0 : a.s;
    switch (a.kind) {
        case Ph::PROJ:
            g.W = P.cp_proj_w; g.N = P.Hc; g.K = P.H; g.pro = Pro::RAW; g.tok = first_tok; g.epi = Epi::BIAS;
            g.bias = P.cp_proj_b; g.dst = P.cx; g.ld_dst = P.Hc; g.dst_buf = BCX;
            break;
        case Ph::QKV:
            // (token assembly) + RMSNorm + q/k/v projection
            g.W = (const char*)B.wqkv + (size_t)l * nqkv * H * e; g.N = nqkv; g.K = H;
            g.pro = Pro::NORM; g.tok = (l == 0 && (a.talker || !proj)) ? first_tok : Tok::NONE; g.epi = Epi::STORE;
            g.src = x; g.src_ld = H; g.src_buf = xb;
            g.norm_w = B.attn_norm + (size_t)l * H; g.dst = P.qkv; g.ld_dst = nqkv; g.dst_buf = BQKV;
            break;
        case Ph::O:
            // O projection + residual
            g.W = (const char*)B.wo + (size_t)l * H * nq * HD * e; g.N = H; g.K = nq * HD;
            g.pro = Pro::LOAD; g.tok = Tok::NONE; g.epi = Epi::ADD; g.src = P.o; g.src_ld = nq * HD; g.src_buf = BO;
            g.dst = x; g.ld_dst = H; g.dst_buf = xb;
            break;
        case Ph::GU:
            // RMSNorm + gate/up + SiLU(g)*u
            g.W = (const char*)B.wgu + (size_t)l * 2 * F * H * e; g.N = F; g.K = H; g.gated = true;
            g.pro = Pro::NORM; g.tok = Tok::NONE; g.epi = Epi::GATED; g.src = x; g.src_ld = H; g.src_buf = xb;
            g.norm_w = B.mlp_norm + (size_t)l * H; g.dst = P.act; g.ld_dst = F; g.dst_buf = BACT;
            break;
        case Ph::DOWN:
            // down projection + residual
            g.W = (const char*)B.wd + (size_t)l * H * F * e; g.N = H; g.K = F;
            g.pro = Pro::LOAD; g.tok = Tok::NONE; g.epi = Epi::ADD; g.src = P.act; g.src_ld = F; g.src_buf = BACT;
            g.dst = x; g.ld_dst = H; g.dst_buf = xb;
            break;
        default:   // HEAD: final norm of the last token -> predictor head[s] / codec head
            g.M = 1; g.pro = Pro::NORM; g.tok = Tok::NONE; g.epi = Epi::STORE;
            g.norm_w = B.final_norm; g.src_ld = H;
            if (a.talker) {
                g.W = P.codec_head; g.N = P.V; g.K = P.H; g.src = P.x; g.src_buf = BX;
                g.dst = P.logits; g.ld_dst = P.V; g.dst_buf = BLOG; g.hout = P.h;
            } else {
                g.W = (const char*)P.cp_heads + (size_t)a.s * P.cpV * P.Hc * e; g.N = P.cpV; g.K = P.Hc;
                g.src = P.cx + (size_t)(M - 1) * P.Hc; g.src_buf = BCX;
                g.dst = P.cpl; g.ld_dst = P.cpV; g.dst_buf = BCPL;
            }
            break;
    }
    return g;
}

template <typename T, class R>
__device__ __forceinline__ void run_phase(R& r, const FrameParams& P, const PhaseAt& a) {
    switch (a.kind) {
        case Ph::ATTN: {
            const bool tk = a.talker;
            const int M = (!tk && a.s == 0) ? 2 : 1;
            const int p0 = tk ? r.talker_pos() : (a.s == 0 ? 0 : a.s + 1);
            r.attention(a.l, tk ? P.t : P.c, M, p0, tk ? P.n_splits : 1, tk);
            break;
        }
        case Ph::DRAW_CP: r.draw_cp(a.s); break;
        case Ph::PREP_T: r.prepare_talker(); break;
        case Ph::DRAW_T: r.draw_talker(); break;
        default: r.gemv(phase_gemv<T>(a, P)); break;
    }
}

// Two walks of the same phase list.  FLAT: one loop, one call site per kind
// of phase, which keeps the large unrolled FMA rows in the instruction cache
// (measured on the 1.7B shape: 3.68 -> 3.08 ms per step).  Nested: a call
// site per phase of a layer, each with its kind known at compile time, so the
// compiler folds the phase's constants into compact tensor-core row code
// (measured on the 0.6B shape: 2.37 ms nested, 2.56 ms flat).
template <typename T, bool FLAT, class R>
__device__ void frame_schedule(R& r, const FrameParams& P) {
    if constexpr (FLAT) {
        const int n = phase_count(P);
        for (int i = 0; i < n && r.live(); ++i) run_phase<T>(r, P, phase_at(i, P));
    } else {
        const bool proj = P.H != P.Hc;
        for (int s = 0; s < P.G - 1 && r.live(); ++s) {
            if (proj) run_phase<T>(r, P, PhaseAt{Ph::PROJ, s, 0, false});
            for (int l = 0; l < P.c.L && r.live(); ++l) {
                run_phase<T>(r, P, PhaseAt{Ph::QKV, s, l, false});
                run_phase<T>(r, P, PhaseAt{Ph::ATTN, s, l, false});
                run_phase<T>(r, P, PhaseAt{Ph::O, s, l, false});
                run_phase<T>(r, P, PhaseAt{Ph::GU, s, l, false});
                run_phase<T>(r, P, PhaseAt{Ph::DOWN, s, l, false});
            }
            run_phase<T>(r, P, PhaseAt{Ph::HEAD, s, 0, false});
            run_phase<T>(r, P, PhaseAt{Ph::DRAW_CP, s, 0, false});
        }
        run_phase<T>(r, P, PhaseAt{Ph::PREP_T, 0, 0, true});
        for (int l = 0; l < P.t.L && r.live(); ++l) {
            run_phase<T>(r, P, PhaseAt{Ph::QKV, 0, l, true});
            run_phase<T>(r, P, PhaseAt{Ph::ATTN, 0, l, true});
            run_phase<T>(r, P, PhaseAt{Ph::O, 0, l, true});
            run_phase<T>(r, P, PhaseAt{Ph::GU, 0, l, true});
            run_phase<T>(r, P, PhaseAt{Ph::DOWN, 0, l, true});
        }
        run_phase<T>(r, P, PhaseAt{Ph::HEAD, 0, 0, true});
        run_phase<T>(r, P, PhaseAt{Ph::DRAW_T, 0, 0, true});
    }
}

template <typename T, int GQ, bool TCR>
__global__ void __launch_bounds__(NTHREADS, 1) frame_kernel(const FrameParams* __restrict__ Pp) {
    extern __shared__ __align__(128) unsigned char smraw[];
    FSmem<T, TCR>& s = *reinterpret_cast<FSmem<T, TCR>*>(smraw);
    const FrameParams& P = *Pp;
    const RowState& rs = P.rows[0];
    if (rs.finished || aborted(P)) return;   // uniform over the grid
    const int frame = rs.sel - 1, pos = rs.pos, code0 = rs.code0;
    // the same checks on every CTA: all leave, or none
    if (frame < 0 || frame >= P.frames_cap || code0 < 0 || code0 >= P.V || rs.sel >= (1 << 22)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(P.err, ERRB_BOUNDS);
        return;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < Ring<TCR>::SLOTS; ++i) { mbar_init(&s.full[i], 1); mbar_init(&s.empty[i], NCW); }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s.codes[0] = code0;
        if (blockIdx.x == 0) P.codes[(size_t)frame * MAX_GROUPS] = code0;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    if (warp == NCW) {
        if ((threadIdx.x & 31) == 0) {
            Producer<T, TCR> pr{s, P};
            pr.pos = pos;
            frame_schedule<T, !TCR>(pr, P);
            pr.drain();
        }
        return;
    }
    Consumer<T, GQ, TCR> c{s, P};
    c.frame = frame;
    c.pos = pos;
    c.base = (unsigned)rs.sel << 10;
    frame_schedule<T, !TCR>(c, P);
}

// ------------------------------------------------------------------ host side
template <typename T, bool TCR>
static size_t smem_for(int xin_bytes) {
    return align128(sizeof(FSmem<T, TCR>)) +
           std::max(2 * align128((size_t)xin_bytes), sizeof(SampSmemT<CP_VMAX>));
}

size_t frame_tile_bytes(bool tc_rows) { return tc_rows ? Ring<true>::TILE : Ring<false>::TILE; }

size_t frame_attn_scratch_bytes() {
    constexpr int GQ = 2;
    return (size_t)(2 * GQ * HD + 4 * HD + 2 * NCW * GQ + NCW * GQ * HD) * sizeof(float);
}

// the kernel variant: fp32 weights (FMA rows), bf16 with FMA rows, bf16 with tensor-core rows
static const void* variant(int dtype, bool tc_rows) {
    if (dtype != Q3_BF16) return (const void*)frame_kernel<float, 2, false>;
    return tc_rows ? (const void*)frame_kernel<bf16, 2, true> : (const void*)frame_kernel<bf16, 2, false>;
}

size_t frame_smem_bytes(int dtype, int xin_bytes, bool tc_rows) {
    const size_t b = dtype != Q3_BF16 ? smem_for<float, false>(xin_bytes)
                   : tc_rows ? smem_for<bf16, true>(xin_bytes) : smem_for<bf16, false>(xin_bytes);
    return b <= 227 * 1024 ? b : 0;
}

cudaError_t frame_setup(int dtype, size_t smem, bool tc_rows) {
    return cudaFuncSetAttribute(variant(dtype, tc_rows), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t frame_occupancy(int dtype, size_t smem, bool tc_rows, int* blocks) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, variant(dtype, tc_rows), NTHREADS, smem);
}

cudaError_t launch_frame(int dtype, bool tc_rows, const FrameParams* params_dev, int grid, size_t smem,
                         cudaStream_t st) {
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
    if (dtype != Q3_BF16) return cudaLaunchKernelEx(&cfg, frame_kernel<float, 2, false>, params_dev);
    if (tc_rows) return cudaLaunchKernelEx(&cfg, frame_kernel<bf16, 2, true>, params_dev);
    return cudaLaunchKernelEx(&cfg, frame_kernel<bf16, 2, false>, params_dev);
}

}  // namespace q3
