// Cluster step kernel: one talker step of a single row in ONE cooperative
// launch of 8 thread-block clusters x 8 CTAs (one cluster per KV head).
//
// What it computes (per frame; Mizuoto "Qwen3-TTS" page, 工作原理 and 速度;
// ncnn discussion 6798 section 1): the code predictor's 2-token prefill
// [h, codec_emb(code0)] and its 14 steps table[s-1](code_s) -> head[s], each
// ending in a draw, then the talker input codec_emb(code0) + sum of the 15
// table rows + the trailing text row, the 28 talker layers and the codec head
// with the codebook-0 selection.
//
// Why clusters.  At batch 1 the step is a chain of ~100 decoder-layer passes;
// what bounds it is the number of dependent cross-SM hand-offs, not the 3.3 GB
// of weights.  A layer here needs two hand-offs through L2 and four inside a
// cluster (distributed shared memory, ~3x cheaper):
//
//   * cluster g owns KV head g: its 8 CTAs compute the 512 q/k/v rows of the
//     head (q heads 2g, 2g+1, k and v head g), all-gather them over DSMEM,
//     and run QK-norm, RoPE and attention without leaving the cluster
//     (predictor: every CTA computes the <= 16-position attention itself from
//     its own shared-memory copy of the head's K/V; talker: positions split
//     over the 8 CTAs, partials all-gathered over DSMEM and merged in rank
//     order);
//   * the O projection is split by K: cluster g multiplies its heads'
//     256-column block, CTA r its 1/8 of the output rows; the 8 clusters'
//     partials of each row slice meet through L2 (epoch-tagged words, summed
//     in cluster order), and the CTAs of a cluster all-gather the new
//     residual over DSMEM;
//   * gate/up rows are split over all 64 CTAs (cluster g: F-slice g);
//     SiLU(g)*u is all-gathered inside the cluster, which then multiplies its
//     F-slice of the down projection (K-split again), reduced like O.
//
// Weights are streamed, not waited for: a producer warp per CTA walks the
// same schedule and copies the CTA's next weight windows (32 KB, one bulk
// copy each) from a packed image into a 3-slot ring ahead of the chain
// (prefetching later windows into L2 as well, PF_WINDOWS > 0, measured
// slower and is compiled out).  The packed image (built once at handle
// creation) stores each CTA's slice of every matrix in mma.m16n8k16 fragment
// order, so a warp reads one 16-byte word per lane per 16x16 weight tile.
// GEMV rows run on the tensor cores: A = 16 weight rows, B = the input's
// bf16 high and low parts (columns 2m, 2m + 1 for token m), fp32 accumulate.
//
// Every wait is bounded (%globaltimer).  A cross-cluster wait that runs out
// sets the TIMEOUT error bit and the abort flag; from then on cross-cluster
// waits return at once, while the weight ring and the cluster-local exchanges
// keep their full protocol, so the launch ends after one more walk of the
// schedule with no copy or peer write still in flight when a CTA leaves.
#include "sampler.cuh"
#include "kernels.h"
#include "cluster_step.h"

#include <algorithm>
#include <cstring>

namespace q3 {
namespace {

constexpr int CS = CL_CS, NCL = CL_NCL, NCTA = CL_NCTA;
constexpr int NCW = 8;                   // consumer warps
constexpr int NT = (NCW + 1) * 32;       // + one producer warp
constexpr int SLOT = 32768;              // ring slot = largest weight window
constexpr int NSLOT = 3;
constexpr int GQ = 2;                    // q heads per KV head
constexpr int QKVR = (GQ + 2) * HD;      // q/k/v rows of one KV head group
constexpr int XMAX = 2048;               // tokens x width of the residual buffer
constexpr int AMAX = 768;                // tokens x F-slice width
constexpr int PATT = GQ * 132;           // one rank's attention partial: per head acc[128], m, l, pad
constexpr int PKV = 16;                  // predictor positions
constexpr int CPV_MAX = 2048;            // predictor vocabulary bound (draw scratch)
constexpr int OPK = 4160;                // operand bf16: 4 x (1024 + 16) or 2 x (2048 + 16)
constexpr int PARTN = 2048;              // K-split partial sums
constexpr int STG = 512;                 // staged outputs
constexpr int XW = 2048;                 // width of a reduction word row
constexpr int TACC = 256;                // talker input slice
constexpr int SIDE = 2048 + 4 * HD;      // per-op vectors: RMSNorm weights [H], q / k norms, RoPE rows
#ifndef PF_WINDOWS
#define PF_WINDOWS 0
#endif
constexpr int PF_AHEAD = PF_WINDOWS;     // weight windows prefetched into L2 ahead of the ring

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ unsigned long long gtime() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ uint32_t cl_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cl_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cl_nclusters() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cl_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t mapa(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
// every thread of every CTA of the cluster (not warp-aligned: the producer
// warp's idle lanes arrive on their own)
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ void mbar_init(uint64_t* b, unsigned n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_expect(uint64_t* b, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
// phase wait for copies into this CTA's own shared memory (ring, side buffers)
__device__ __forceinline__ bool mbar_try_cta(uint64_t* b, unsigned par) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(su32(b)), "r"(par) : "memory");
    return ok != 0;
}
// phase wait that also acquires peer CTAs' writes (DSMEM all-gathers)
__device__ __forceinline__ bool mbar_try(uint64_t* b, unsigned par) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(su32(b)), "r"(par) : "memory");
    return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* b) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(su32(dst)), "l"(src), "r"(bytes), "r"(su32(b)) : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
// 16 bytes into a peer's shared memory, completing tx bytes on the peer's mbarrier
__device__ __forceinline__ void st_async4(uint32_t raddr, float4 v, uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
                 ::"r"(raddr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(rbar) : "memory");
}
// barrier of the 256 consumer threads that also ORs a flag over them
__device__ __forceinline__ bool bar_or(bool v) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.or.pred q, 2, 256, p;\n\t"
        "selp.s32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((int)v)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(a));
    return r;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 r;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(a));
    return r;
}
// D += A B, mma.m16n8k16 bf16 -> fp32; A = 16 weight rows (one 16-byte word a
// lane), B = this lane's operand column
__device__ __forceinline__ void mma16(float (&d)[4], const uint4& a, const uint2& b) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y));
}
__device__ __forceinline__ Word ld_word(const Word* p) {
    Word w;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p));
    return w;
}
__device__ __forceinline__ void st_word(Word* p, float v, unsigned ep) {
    const Word w = ((Word)ep << 32) | (Word)__float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w));
}
__device__ __forceinline__ unsigned ep_of(Word w) { return (unsigned)(w >> 32); }
__device__ __forceinline__ float val_of(Word w) { return __uint_as_float((unsigned)w); }

// position of element j (0..15) of a 16-element K step in the operand buffer:
// lane q of a fragment reads elements 2q, 2q+1, 2q+8, 2q+9 as 4 consecutive ones
__device__ __forceinline__ int perm16(int k) {
    const int j = k & 15;
    return (k & ~15) + 4 * ((j & 7) >> 1) + 2 * (j >> 3) + (j & 1);
}

// ------------------------------------------------------------------ shared memory
struct Work {
    bf16 op[OPK];                 // GEMV operand: [2M][K + 16] bf16 high/low, K order permuted
    float part[PARTN];            // K-split partial sums [block][split][16][M]
    float stage[STG];             // a phase's outputs before they leave the CTA
    float o[2 * GQ * HD];         // attention output [M][256]
    float q[2 * GQ * HD];         // q after QK-norm and RoPE [M][2][128]
    float kv[2 * 2 * HD];         // new k, v (cache precision) [M][2][128]
    float wacc[NCW * PATT];       // talker attention: per-warp partials
    float red[NCW * 4];
    float rs[4];                  // RMSNorm scale per token
};
struct __align__(128) Sm {
    unsigned char ring[NSLOT][SLOT];
    bf16 pkv[CL_MAX_CP_LAYERS][2][PKV][HD];   // predictor K/V of this cluster's head
    float qkv[2 * QKVR];          // DSMEM: q/k/v rows of the head group [M][512]
    float x[XMAX];                // DSMEM: residual [M][width]
    float a[AMAX];                // DSMEM: SiLU(g)*u of the cluster's F-slice [M][Fc]
    float patt[CS * PATT];        // DSMEM: talker attention partials [rank][head][132]
    union {
        Work w;
        SampSmemT<CPV_MAX> draw;  // predictor draw scratch (the Work buffers are idle then)
    } u;
    float tacc[TACC];             // this CTA's slice of the next talker input
    float side[2][SIDE];          // per-op vectors, copied ahead by the producer
    uint64_t full[NSLOT], empty[NSLOT];
    uint64_t side_full[2], side_empty[2];
    uint64_t bar_qkv, bar_x, bar_a, bar_patt;
    int codes[MAX_GROUPS];
};

// ------------------------------------------------------------------ schedule
enum OpKind : int { OP_PROJ, OP_QKV, OP_ATT, OP_O, OP_GU, OP_DOWN, OP_HEADC, OP_TIN, OP_HEADT };
struct Op {
    int kind, s, l;
    bool talker;
};

__device__ __forceinline__ int n_ops(const ClParams& P) {
    const int proj = P.H != P.Hc ? 1 : 0;
    return (P.G - 1) * (proj + 5 * P.Lc + 1) + 1 + 5 * P.Lt + 1;
}
__device__ __forceinline__ Op op_at(int i, const ClParams& P) {
    const int proj = P.H != P.Hc ? 1 : 0;
    const int per = proj + 5 * P.Lc + 1;
    const int npred = (P.G - 1) * per;
    Op o{OP_TIN, 0, 0, false};
    if (i < npred) {
        o.s = i / per;
        int j = i - o.s * per;
        if (proj && j == 0) { o.kind = OP_PROJ; return o; }
        j -= proj;
        if (j < 5 * P.Lc) { o.l = j / 5; o.kind = OP_QKV + j % 5; }
        else o.kind = OP_HEADC;
        return o;
    }
    o.talker = true;
    int j = i - npred;
    if (j == 0) return o;
    j -= 1;
    if (j < 5 * P.Lt) { o.l = j / 5; o.kind = OP_QKV + j % 5; }
    else o.kind = OP_HEADT;
    return o;
}

// The GEMV of an op: this CTA's packed slice, its rows and K.
struct Gv {
    const unsigned char* src;
    int R, K;
    bool ok;
};
__device__ __forceinline__ Gv gemv_of(const Op& o, const ClParams& P, int cta) {
    const ClLayout& L = P.lay;
    const int H = o.talker ? P.H : P.Hc, F = o.talker ? P.F : P.Fc;
    Gv g{nullptr, 0, 0, true};
    size_t off = 0, per = 0;
    const size_t* offs = o.talker ? L.off_t : L.off_c;
    const size_t* pers = o.talker ? L.per_t : L.per_c;
    switch (o.kind) {
        case OP_QKV: g.R = QKVR / CS; g.K = H; off = offs[0]; per = pers[0]; break;
        case OP_O: g.R = H / CS; g.K = GQ * HD; off = offs[1]; per = pers[1]; break;
        case OP_GU: g.R = 2 * (F / NCL) / CS; g.K = H; off = offs[2]; per = pers[2]; break;
        case OP_DOWN: g.R = H / CS; g.K = F / NCL; off = offs[3]; per = pers[3]; break;
        case OP_HEADC:
            g.R = P.cpV / NCTA; g.K = P.Hc; off = L.off_cph + (size_t)o.s * L.per_cph; per = 0; break;
        case OP_HEADT: g.R = P.V / NCTA; g.K = P.H; off = L.off_th; per = 0; break;
        case OP_PROJ: g.R = P.Hc / CS; g.K = P.H / NCL; off = L.off_proj; per = 0; break;
        default: g.ok = false; return g;
    }
    const size_t slice = (size_t)g.R * g.K * 2;
    g.src = P.pack + off + (size_t)o.l * per + (size_t)cta * slice;
    return g;
}

// How a slice is cut into ring windows.  Blocks are 16 rows x K (K/16 steps of
// 512 bytes).  A: blocks no larger than a slot; wb blocks per window, S K
// splits per block (wb * S <= 8 units, one per warp).  B: a block larger than
// a slot; windows of 64 K steps, each warp takes 1/8 of every window and keeps
// its sum across the block's windows (S = 8).
struct Win {
    int nb, nks, bb, wb, S, wpb, nwin;
};
__device__ __forceinline__ Win win_of(int R, int K) {
    Win w;
    w.nb = R / 16;
    w.nks = K / 16;
    w.bb = w.nks * 512;
    if (w.bb <= SLOT) {
        w.wb = min(min(w.nb, SLOT / w.bb), NCW);
        w.S = max(1, NCW / w.wb);
        w.wpb = 1;
        w.nwin = (w.nb + w.wb - 1) / w.wb;
    } else {
        w.wb = 1;
        w.S = NCW;
        w.wpb = (w.nks + SLOT / 512 - 1) / (SLOT / 512);
        w.nwin = w.nb * w.wpb;
    }
    return w;
}
// byte range of window i inside the slice
__device__ __forceinline__ void win_range(const Win& w, int i, int& off, int& bytes) {
    if (w.wpb == 1) {
        const int b0 = i * w.wb, b1 = min(w.nb, b0 + w.wb);
        off = b0 * w.bb;
        bytes = (b1 - b0) * w.bb;
    } else {
        const int b = i / w.wpb, kr = i - b * w.wpb;
        const int k0 = kr * (SLOT / 512), k1 = min(w.nks, k0 + SLOT / 512);
        off = b * w.bb + k0 * 512;
        bytes = (k1 - k0) * 512;
    }
}

// The per-op vectors an op reads (copied into a side buffer ahead of it): the
// RMSNorm weights of q/k/v, gate/up and the heads; q/k/v also carries the
// layer's q and k norm weights and the RoPE rows of its token positions.
struct SideSrc {
    const float* norm;
    int H;
    const float* qn;
    const float* kn;
    const float2* rope;
    int rows;
};
__device__ __forceinline__ bool side_of(const Op& o, const ClParams& P, int pos, SideSrc& d) {
    const int H = o.talker ? P.H : P.Hc;
    d = SideSrc{nullptr, H, nullptr, nullptr, nullptr, 0};
    if (o.kind == OP_QKV) {
        d.norm = (o.talker ? P.t_attn_norm : P.c_attn_norm) + (size_t)o.l * H;
        d.qn = (o.talker ? P.t_q_norm : P.c_q_norm) + (size_t)o.l * HD;
        d.kn = (o.talker ? P.t_k_norm : P.c_k_norm) + (size_t)o.l * HD;
        const int p0 = o.talker ? pos : (o.s == 0 ? 0 : o.s + 1);
        d.rope = P.rope + (size_t)p0 * (HD / 2);
        d.rows = (!o.talker && o.s == 0) ? 2 : 1;
        return true;
    }
    if (o.kind == OP_GU) { d.norm = (o.talker ? P.t_mlp_norm : P.c_mlp_norm) + (size_t)o.l * H; return true; }
    if (o.kind == OP_HEADC) { d.norm = P.c_final_norm; return true; }
    if (o.kind == OP_HEADT) { d.norm = P.t_final_norm; return true; }
    return false;
}
// offsets of the pieces in a side buffer (floats)
__device__ __forceinline__ int side_qn(int H) { return H; }
__device__ __forceinline__ int side_kn(int H) { return H + HD; }
__device__ __forceinline__ int side_rope(int H) { return H + 2 * HD; }

// Cached talker positions [j0, j1) (before the new token at pos) of rank r's
// split, and whether they fit one ring slot.
__device__ __forceinline__ void talker_split(int pos, int r, int& j0, int& j1) {
    const int n = pos + 1;
    const int chunk = (n + CS - 1) / CS;
    j0 = min(n, r * chunk);
    j1 = min(n, j0 + chunk);
}
__device__ __forceinline__ bool kv_prefetch(int pos, int r, int& c0, int& c1) {
    int j0, j1;
    talker_split(pos, r, j0, j1);
    c0 = j0;
    c1 = min(j1, pos);
    return c1 > c0 && (c1 - c0) * HD * 2 * 2 <= SLOT;
}

__device__ __forceinline__ bool aborted(const ClParams& P) { return *(volatile unsigned*)&P.ctl[0] != 0u; }
__device__ __forceinline__ void raise_abort(const ClParams& P, int bits) {
    if (bits) atomicOr(P.err, bits);
    atomicExch(&P.ctl[0], 1u);
}

// ------------------------------------------------------------------ producer
struct Producer {
    Sm& s;
    const ClParams& P;
    int cta, rank;
    int pos;
    unsigned seq = 0;
    unsigned sseq = 0;   // side buffers filled
    bool ok = true;

    // the op's vectors into the next side buffer
    __device__ __forceinline__ bool side(const Op& o) {
        SideSrc d;
        if (!side_of(o, P, pos, d)) return true;
        const int slot = (int)(sseq & 1);
        if (sseq >= 2) {
            const unsigned par = ((sseq >> 1) - 1) & 1;
            const unsigned long long t0 = gtime();
            unsigned it = 0;
            while (!mbar_try_cta(&s.side_empty[slot], par)) {
                __nanosleep(200);   // the producer waits most of the time: leave the issue slots to the consumers
                if ((++it & 15u) == 0 && gtime() - t0 > 4ull * (unsigned long long)P.wait_ns) { ok = false; return false; }
            }
        }
        ++sseq;
        float* b = s.side[slot];
        unsigned bytes = (unsigned)(d.H * 4);
        if (d.qn) bytes += 2 * HD * 4 + (unsigned)d.rows * HD * 4;
        mbar_expect(&s.side_full[slot], bytes);
        bulk_g2s(b, d.norm, (unsigned)(d.H * 4), &s.side_full[slot]);
        if (d.qn) {
            bulk_g2s(b + side_qn(d.H), d.qn, HD * 4, &s.side_full[slot]);
            bulk_g2s(b + side_kn(d.H), d.kn, HD * 4, &s.side_full[slot]);
            bulk_g2s(b + side_rope(d.H), d.rope, (unsigned)d.rows * HD * 4, &s.side_full[slot]);
        }
        return true;
    }

    __device__ __forceinline__ bool take(int& slot) {
        slot = (int)(seq % NSLOT);
        if (seq >= (unsigned)NSLOT) {
            const unsigned par = ((seq / NSLOT) - 1) & 1;
            if (!mbar_try_cta(&s.empty[slot], par)) {
                const unsigned long long t0 = gtime();
                unsigned it = 0;
                while (!mbar_try_cta(&s.empty[slot], par)) {
                    __nanosleep(200);   // see side(): back off while the ring is full
                    if ((++it & 15u) == 0 && gtime() - t0 > 4ull * (unsigned long long)P.wait_ns) {
                        ok = false;
                        return false;
                    }
                }
            }
        }
        ++seq;
        return true;
    }
    // L2 prefetch cursor: the window PF_AHEAD windows past the last one issued
    int pf_op = 0, pf_win = 0;
    unsigned pf_seq = 0;
    __device__ __forceinline__ void prefetch_to(unsigned target, int nops) {
        while (pf_seq < target && pf_op < nops) {
            const Gv g = gemv_of(op_at(pf_op, P), P, cta);
            if (!g.ok) { ++pf_op; pf_win = 0; continue; }
            const Win w = win_of(g.R, g.K);
            if (pf_win >= w.nwin) { ++pf_op; pf_win = 0; continue; }
            int off, bytes;
            win_range(w, pf_win, off, bytes);
            prefetch_l2(g.src + off, (unsigned)bytes);
            ++pf_win;
            ++pf_seq;
        }
    }
    __device__ __forceinline__ void run() {
        const int nops = n_ops(P);
        unsigned wseq = 0;   // weight windows issued
        for (int i = 0; i < nops && ok; ++i) {
            const Op o = op_at(i, P);
            if (!side(o)) return;
            if (o.kind == OP_ATT) {
                int c0, c1;
                if (!o.talker || !kv_prefetch(pos, rank, c0, c1)) continue;
                int slot;
                if (!take(slot)) return;
                const size_t row = (size_t)HD * 2;
                const size_t base = (((size_t)o.l * P.max_batch) * NCL + cl_id()) * P.cap + c0;
                const unsigned bytes = (unsigned)((c1 - c0) * row);
                mbar_expect(&s.full[slot], 2 * bytes);
                bulk_g2s(s.ring[slot], (const char*)P.Kc + base * row, bytes, &s.full[slot]);
                bulk_g2s(s.ring[slot] + bytes, (const char*)P.Vc + base * row, bytes, &s.full[slot]);
                continue;
            }
            const Gv g = gemv_of(o, P, cta);
            if (!g.ok) continue;
            const Win w = win_of(g.R, g.K);
            for (int k = 0; k < w.nwin; ++k) {
                int off, bytes, slot;
                win_range(w, k, off, bytes);
                if (PF_AHEAD > 0) prefetch_to(wseq + PF_AHEAD + 1, nops);
                ++wseq;
                if (!take(slot)) return;
                mbar_expect(&s.full[slot], (unsigned)bytes);
                bulk_g2s(s.ring[slot], g.src + off, (unsigned)bytes, &s.full[slot]);
            }
        }
    }
    // copies issued and not consumed must land before the CTA exits
    __device__ __forceinline__ void drain() {
        for (unsigned t = (sseq > 2u ? sseq - 2 : 0); t < sseq; ++t) {
            const unsigned long long t0 = gtime();
            while (!mbar_try_cta(&s.side_full[t & 1], (t >> 1) & 1))
                if (gtime() - t0 > (unsigned long long)P.wait_ns) break;
        }
        for (unsigned t = (seq > (unsigned)NSLOT ? seq - NSLOT : 0); t < seq; ++t) {
            const unsigned long long t0 = gtime();
            while (!mbar_try_cta(&s.full[t % NSLOT], (t / NSLOT) & 1))
                if (gtime() - t0 > (unsigned long long)P.wait_ns) break;
        }
    }
};

// ------------------------------------------------------------------ consumer
struct Consumer {
    Sm& s;
    const ClParams& P;
    int cta, g, rank;
    int frame, pos;
    unsigned base;          // epoch of this launch's exchange 0
    unsigned gex = 0;       // global exchanges done
    unsigned xr_cnt = 0;    // reductions done (word buffer parity)
    unsigned rseq = 0;      // ring windows consumed
    unsigned n_qkv = 0, n_x = 0, n_a = 0, n_patt = 0;   // DSMEM buffer uses
    unsigned head_cnt = 0;
    unsigned sseq = 0;      // side buffers consumed
    int qkv_side = 0;       // side buffer of the last q/k/v op (read again by its attention)
    bool fail = false;      // a wait of this thread gave up (launch is aborting)

    __device__ __forceinline__ unsigned next_epoch() { return base + (++gex); }
    // barrier of the consumer threads; a failed wait of any thread becomes known to all
    __device__ __forceinline__ void sync() { fail = bar_or(fail); }

    // -------- waits
    template <bool CLUSTER = false>
    __device__ __forceinline__ bool wait_mbar(uint64_t* b, unsigned par) {
        if (CLUSTER ? mbar_try(b, par) : mbar_try_cta(b, par)) return true;
        const unsigned long long t0 = gtime();
        unsigned it = 0;
        while (!(CLUSTER ? mbar_try(b, par) : mbar_try_cta(b, par))) {
            if ((++it & 63u) == 0 && gtime() - t0 > 2ull * (unsigned long long)P.wait_ns) {
                raise_abort(P, ERRB_TIMEOUT);
                fail = true;
                return false;
            }
        }
        return true;
    }
    // poll N words until each carries epoch e; in abort mode return at once
    template <int N>
    __device__ __forceinline__ void poll(Word (&w)[N], const Word* const (&p)[N], unsigned e) {
#pragma unroll
        for (int j = 0; j < N; ++j) w[j] = ld_word(p[j]);
        unsigned long long t0 = 0;
        for (unsigned it = 0;; ++it) {
            bool pend = false;
#pragma unroll
            for (int j = 0; j < N; ++j) pend |= ep_of(w[j]) != e;
            if (!pend || fail) return;
            if (it == 0) t0 = gtime();
            if ((it & 31u) == 31u) {
                if (aborted(P)) { fail = true; return; }
                if (gtime() - t0 > (unsigned long long)P.wait_ns) {
                    raise_abort(P, ERRB_TIMEOUT);
                    fail = true;
                    return;
                }
            }
#pragma unroll
            for (int j = 0; j < N; ++j)
                if (ep_of(w[j]) != e) w[j] = ld_word(p[j]);
        }
    }

    // -------- operand
    // token m's value at k (hi, lo) into the permuted operand rows 2m, 2m+1
    __device__ __forceinline__ void put_op(int m, int K, int k, float v) {
        const int KP = K + 16;
        const bf16 hi = __float2bfloat16_rn(v);
        const bf16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
        s.u.w.op[(2 * m) * KP + perm16(k)] = hi;
        s.u.w.op[(2 * m + 1) * KP + perm16(k)] = lo;
    }
    // operand x (.) w of M tokens of src (smem [M][K]); r_m = rsqrt(mean(x^2) + eps) into rs[m]
    // the op's side buffer (waits for it; returns its index)
    __device__ __forceinline__ int side_take() {
        const int slot = (int)(sseq & 1);
        const unsigned par = (sseq >> 1) & 1;
        ++sseq;
        wait_mbar(&s.side_full[slot], par);
        return slot;
    }
    __device__ __forceinline__ void side_release(int slot) {
        __syncwarp();   // every lane of the warp is done with the buffer
        if ((threadIdx.x & 31) == 0) mbar_arrive(&s.side_empty[slot]);
    }
    // w: the RMSNorm weights (shared memory)
    __device__ __forceinline__ void build_norm(const float* src, int M, int K, const float* w) {
        const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
        float ss[2] = {0.f, 0.f};
        for (int m = 0; m < M; ++m)
            for (int k = tid; k < K; k += 256) {
                const float v = src[m * K + k];
                ss[m] = fmaf(v, v, ss[m]);
                put_op(m, K, k, v * w[k]);
            }
        for (int m = 0; m < M; ++m) {
            const float t = warp_sum(ss[m]);
            if (lane == 0) s.u.w.red[warp * 4 + m] = t;
        }
        sync();
        if (tid < M) {
            float t = 0.f;
            for (int i = 0; i < NCW; ++i) t += s.u.w.red[i * 4 + tid];
            s.u.w.rs[tid] = 1.0f / sqrtf(t / (float)K + P.eps);
        }
        // the GEMV's barrier orders rs before its readers
    }
    __device__ __forceinline__ void build_plain(const float* src, int ld, int M, int K) {
        for (int m = 0; m < M; ++m)
            for (int k = threadIdx.x; k < K; k += 256) put_op(m, K, k, src[m * ld + k]);
    }

    // -------- the GEMV: raw dot products into part[]; one barrier before, one after
    __device__ __forceinline__ void mma_steps(uint32_t a, uint32_t b, bool bl, int nk, float (&d)[4]) {
        float e[4] = {0.f, 0.f, 0.f, 0.f};
        int k = 0;
        for (; k + 2 <= nk; k += 2) {
            const uint4 A0 = lds128(a), A1 = lds128(a + 512);
            uint2 B0 = make_uint2(0u, 0u), B1 = make_uint2(0u, 0u);
            if (bl) { B0 = lds64(b); B1 = lds64(b + 32); }
            mma16(d, A0, B0);
            mma16(e, A1, B1);
            a += 1024;
            b += 64;
        }
        if (k < nk) {
            const uint4 A0 = lds128(a);
            uint2 B0 = make_uint2(0u, 0u);
            if (bl) B0 = lds64(b);
            mma16(d, A0, B0);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) d[i] += e[i];
    }
    __device__ __forceinline__ void flush(const float (&d)[4], int blk, int split, int S, int M) {
        const int lane = threadIdx.x & 31, gq = lane >> 2, q = lane & 3;
        if (q < M) {
            float* p = s.u.w.part + ((size_t)(blk * S + split) * 16) * M;
            p[gq * M + q] = d[0] + d[1];
            p[(gq + 8) * M + q] = d[2] + d[3];
        }
    }
    __device__ __forceinline__ void gemv(const Gv& gv, int M) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const Win w = win_of(gv.R, gv.K);
        const int KP = gv.K + 16;
        const bool bl = (lane >> 2) < 2 * M;
        const uint32_t opb = su32(s.u.w.op) + (uint32_t)(((lane >> 2) * KP + 4 * (lane & 3)) * 2);
        sync();   // operand complete
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int i = 0; i < w.nwin; ++i) {
            const int slot = (int)(rseq % NSLOT);
            const unsigned par = (rseq / NSLOT) & 1;
            ++rseq;
            // every window is waited for, also while the launch aborts (a slot is
            // refilled only after its copy landed); warp-uniform for the MMAs
            const bool have = __all_sync(0xffffffffu, wait_mbar(&s.full[slot], par));
            const uint32_t sb = su32(s.ring[slot]) + (uint32_t)lane * 16;
            if (have) {
                if (w.wpb == 1) {
                    const int b0 = i * w.wb, nbw = min(w.nb, b0 + w.wb) - b0;
                    if (warp < nbw * w.S) {
                        const int bl_i = warp / w.S, j = warp - bl_i * w.S;
                        const int k0 = w.nks * j / w.S, k1 = w.nks * (j + 1) / w.S;
                        float d[4] = {0.f, 0.f, 0.f, 0.f};
                        mma_steps(sb + (uint32_t)(bl_i * w.bb + k0 * 512), opb + (uint32_t)(k0 * 32), bl, k1 - k0, d);
                        flush(d, b0 + bl_i, j, w.S, M);
                    }
                } else {
                    const int b = i / w.wpb, kr = i - b * w.wpb;
                    const int lo = kr * (SLOT / 512), hi = min(w.nks, lo + SLOT / 512), n = hi - lo;
                    const int k0 = lo + n * warp / NCW, k1 = lo + n * (warp + 1) / NCW;
                    mma_steps(sb + (uint32_t)((k0 - lo) * 512), opb + (uint32_t)(k0 * 32), bl, k1 - k0, acc);
                    if (kr == w.wpb - 1) {
                        flush(acc, b, warp, w.S, M);
#pragma unroll
                        for (int t = 0; t < 4; ++t) acc[t] = 0.f;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.empty[slot]);
        }
        sync();   // partials complete
    }
    // sum of the K splits of row i, token m (fixed order)
    __device__ __forceinline__ float gsum(const Gv& gv, int i, int m, int M) {
        const Win w = win_of(gv.R, gv.K);
        const float* p = s.u.w.part + ((size_t)((i >> 4) * w.S) * 16 + (i & 15)) * M + m;
        float v = 0.f;
        for (int j = 0; j < w.S; ++j) v += p[(size_t)j * 16 * M];
        return fail ? 0.f : v;
    }

    // -------- DSMEM all-gather: this CTA's n floats of token m (stage[m*n ..]) go
    // to offset m * width + rank * n of buffer `dst` in every CTA of the cluster
    __device__ __forceinline__ void ag_send(const float* src, int M, int n, float* dst, int width, uint64_t* bar, unsigned total) {
        if (threadIdx.x == 0) mbar_expect(bar, total);
        const int n4 = n / 4;
        const int sends = M * n4 * CS;
        const uint32_t bar_l = su32(bar);
        for (int t = threadIdx.x; t < sends; t += 256) {
            const int peer = t / (M * n4), rem = t - peer * (M * n4);
            const int m = rem / n4, j = rem - m * n4;
            const float4 v = *reinterpret_cast<const float4*>(src + m * n + 4 * j);
            const uint32_t la = su32(dst + m * width + rank * n + 4 * j);
            st_async4(mapa(la, (uint32_t)peer), v, mapa(bar_l, (uint32_t)peer));
        }
    }
    __device__ __forceinline__ void ag_wait(uint64_t* bar, unsigned& cnt) {
        const unsigned par = cnt & 1;
        ++cnt;
        wait_mbar<true>(bar, par);
    }

    // -------- cross-cluster reduction of stage[m*R + i] (rows row0.., width W),
    // plus base (residual x or bias), result all-gathered into s.x [M][W]
    __device__ __forceinline__ void reduce_x(int M, int R, int W, bool residual, const float* bias) {
        const unsigned e = next_epoch();
        const int par = (int)(xr_cnt++ & 1);
        Word* buf = P.xr + (size_t)par * NCL * 2 * XW;
        const int row0 = rank * R;
        float* st = s.u.w.stage;
        const bool skip = P.inject_skip >= 0 && cta == 0 && (int)gex == P.inject_skip;
        for (int t = threadIdx.x; t < M * R; t += 256) {
            const int m = t / R, i = t - m * R;
            if (!skip) st_word(buf + ((size_t)g * 2 + m) * XW + row0 + i, st[t], e);
        }
        for (int t = threadIdx.x; t < M * R; t += 256) {
            const int m = t / R, i = t - m * R;
            const Word* p[NCL];
#pragma unroll
            for (int c = 0; c < NCL; ++c) p[c] = buf + ((size_t)c * 2 + m) * XW + row0 + i;
            Word w[NCL];
            poll<NCL>(w, p, e);
            float acc = residual ? s.x[m * W + row0 + i] : (bias ? __ldg(bias + row0 + i) : 0.f);
#pragma unroll
            for (int c = 0; c < NCL; ++c) acc += val_of(w[c]);
            st[t] = acc;
        }
        sync();
        ag_send(st, M, R, s.x, W, &s.bar_x, (unsigned)(M * W * 4));
        ag_wait(&s.bar_x, n_x);
    }

    // -------- ops
    __device__ __forceinline__ int tokens(const Op& o) const { return (!o.talker && o.s == 0) ? 2 : 1; }

    // predictor input tokens of pass s (talker width) -> s.x (no projection)
    // or the projection operand (cluster's column slice)
    __device__ __forceinline__ float token_val(int s_, int m, int i) {
        const bf16* ce = (const bf16*)P.codec_emb;
        const bf16* te = (const bf16*)P.cp_emb;
        if (s_ == 0) return m == 0 ? __ldcg(P.h + i) : __bfloat162float(ce[(size_t)s.codes[0] * P.H + i]);
        return __bfloat162float(te[((size_t)(s_ - 1) * P.cpV + s.codes[s_]) * P.H + i]);
    }
    __device__ __forceinline__ void tacc_add_table(int s_) {
        // table[s-1](code_s) joins the next talker input (sum order: codec, tables 1..15, text)
        if (s_ < 1) return;
        const int Rt = P.H / CS;
        const bf16* te = (const bf16*)P.cp_emb + ((size_t)(s_ - 1) * P.cpV + s.codes[s_]) * P.H + rank * Rt;
        for (int i = threadIdx.x; i < Rt; i += 256) s.tacc[i] += __bfloat162float(te[i]);
    }

    // QK-norm + RoPE of q heads and k, v rounded to the cache precision
    __device__ __forceinline__ void att_prep(const Op& o, int M, int p0) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int H = o.talker ? P.H : P.Hc;
        const float* sd = s.side[qkv_side];
        const float* qn = sd + side_qn(H);
        const float* kn = sd + side_kn(H);
        const float2* rope = reinterpret_cast<const float2*>(sd + side_rope(H));
        if (warp < 4 * M) {
            const int m = warp >> 2, u = warp & 3;   // u: q0, q1, k, v
            const float* src = s.qkv + m * QKVR + u * HD;
            float e[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) e[i] = src[lane + 32 * i];
            if (u < 3) {
                const float* wn = u < 2 ? qn : kn;
                const float ss = warp_sum(e[0] * e[0] + e[1] * e[1] + e[2] * e[2] + e[3] * e[3]);
                const float r = 1.0f / sqrtf(ss / (float)HD + P.eps);
#pragma unroll
                for (int i = 0; i < 4; ++i) e[i] = e[i] * r * wn[lane + 32 * i];
                const float2 c0 = rope[m * (HD / 2) + lane];
                const float2 c1 = rope[m * (HD / 2) + lane + 32];
                float a = e[0], b = e[2];
                e[0] = a * c0.x - b * c0.y; e[2] = b * c0.x + a * c0.y;
                a = e[1]; b = e[3];
                e[1] = a * c1.x - b * c1.y; e[3] = b * c1.x + a * c1.y;
            }
            if (u < 2) {
#pragma unroll
                for (int i = 0; i < 4; ++i) s.u.w.q[(m * GQ + u) * HD + lane + 32 * i] = e[i];
            } else {
                const int kv = u - 2;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const bf16 hb = __float2bfloat16_rn(e[i]);
                    s.u.w.kv[(m * 2 + kv) * HD + lane + 32 * i] = __bfloat162float(hb);
                    if (!o.talker) s.pkv[o.l][kv][p0 + m][lane + 32 * i] = hb;
                }
                if (o.talker && rank == 0) {
                    // the new token's k / v into the talker cache (read by later steps)
                    bf16* dstp = (bf16*)(kv == 0 ? P.Kc : P.Vc) +
                                 ((((size_t)o.l * P.max_batch) * NCL + g) * P.cap + pos) * HD;
#pragma unroll
                    for (int i = 0; i < 4; ++i) dstp[lane + 32 * i] = __float2bfloat16_rn(e[i]);
                }
            }
        }
        sync();
        side_release(qkv_side);
    }

    // predictor attention: every CTA, positions 0..p0+m from its own cache copy
    __device__ __forceinline__ void att_pred(const Op& o, int M, int p0) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        if (warp < 2 * M) {
            const int m = warp >> 1, hh = warp & 1;
            const int np = p0 + m + 1;
            const float* q = s.u.w.q + (m * GQ + hh) * HD + 4 * lane;
            const float q0 = q[0], q1 = q[1], q2 = q[2], q3 = q[3];
            float sc[PKV];
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < PKV; ++j) {
                if (j < np) {
                    const uint2 kk = *reinterpret_cast<const uint2*>(&s.pkv[o.l][0][j][4 * lane]);
                    float d = q0 * __uint_as_float(kk.x << 16);
                    d = fmaf(q1, __uint_as_float(kk.x & 0xffff0000u), d);
                    d = fmaf(q2, __uint_as_float(kk.y << 16), d);
                    d = fmaf(q3, __uint_as_float(kk.y & 0xffff0000u), d);
                    sc[j] = warp_sum(d) * 0.08838834764831845f;
                    mx = fmaxf(mx, sc[j]);
                }
            }
            float den = 0.f, a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int j = 0; j < PKV; ++j) {
                if (j < np) {
                    const float p = expf(sc[j] - mx);
                    den += p;
                    const uint2 vv = *reinterpret_cast<const uint2*>(&s.pkv[o.l][1][j][4 * lane]);
                    a0 = fmaf(p, __uint_as_float(vv.x << 16), a0);
                    a1 = fmaf(p, __uint_as_float(vv.x & 0xffff0000u), a1);
                    a2 = fmaf(p, __uint_as_float(vv.y << 16), a2);
                    a3 = fmaf(p, __uint_as_float(vv.y & 0xffff0000u), a3);
                }
            }
            float* out = s.u.w.o + m * (GQ * HD) + hh * HD + 4 * lane;
            out[0] = a0 / den; out[1] = a1 / den; out[2] = a2 / den; out[3] = a3 / den;
        }
        sync();
    }

    // talker attention: rank r covers its split of positions 0..pos; partials
    // all-gathered over DSMEM and merged in rank order by every CTA
    __device__ __forceinline__ void att_talker(const Op& o) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
        int j0, j1, c0, c1;
        talker_split(pos, rank, j0, j1);
        const bool pre = kv_prefetch(pos, rank, c0, c1);
        const bf16* kr = nullptr;
        const bf16* vr = nullptr;
        int slot = -1;
        bool have = true;
        if (pre) {
            slot = (int)(rseq % NSLOT);
            const unsigned par = (rseq / NSLOT) & 1;
            ++rseq;
            have = __all_sync(0xffffffffu, wait_mbar(&s.full[slot], par));
            kr = reinterpret_cast<const bf16*>(s.ring[slot]);
            vr = kr + (size_t)(c1 - c0) * HD;
        }
        const bf16* Kg = (const bf16*)P.Kc + ((((size_t)o.l * P.max_batch) * NCL + g) * P.cap) * HD;
        const bf16* Vg = (const bf16*)P.Vc + ((((size_t)o.l * P.max_batch) * NCL + g) * P.cap) * HD;
        const float* q0p = s.u.w.q;
        const float* q1p = s.u.w.q + HD;
        float mx[GQ] = {-INFINITY, -INFINITY}, ls[GQ] = {0.f, 0.f}, acc[GQ][4] = {};
        for (int j = j0 + warp; j < j1 && have; j += NCW) {
            float kk[4], vv[4];
            if (j == pos) {
#pragma unroll
                for (int i = 0; i < 4; ++i) { kk[i] = s.u.w.kv[lane + 32 * i]; vv[i] = s.u.w.kv[HD + lane + 32 * i]; }
            } else if (pre && j >= c0 && j < c1) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    kk[i] = __bfloat162float(kr[(size_t)(j - c0) * HD + lane + 32 * i]);
                    vv[i] = __bfloat162float(vr[(size_t)(j - c0) * HD + lane + 32 * i]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    kk[i] = __bfloat162float(__ldcg(Kg + (size_t)j * HD + lane + 32 * i));
                    vv[i] = __bfloat162float(__ldcg(Vg + (size_t)j * HD + lane + 32 * i));
                }
            }
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) {
                const float* q = hh ? q1p : q0p;
                float d = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) d = fmaf(q[lane + 32 * i], kk[i], d);
                d = warp_sum(d) * 0.08838834764831845f;
                const float mn = fmaxf(mx[hh], d);
                const float c = expf(mx[hh] - mn);
                const float p = expf(d - mn);
                ls[hh] = ls[hh] * c + p;
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[hh][i] = fmaf(p, vv[i], acc[hh][i] * c);
                mx[hh] = mn;
            }
        }
        __syncwarp();
        if (slot >= 0 && lane == 0) mbar_arrive(&s.empty[slot]);
        float* wa = s.u.w.wacc + warp * PATT;
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
#pragma unroll
            for (int i = 0; i < 4; ++i) wa[hh * 132 + lane + 32 * i] = acc[hh][i];
            if (lane == 0) { wa[hh * 132 + HD] = mx[hh]; wa[hh * 132 + HD + 1] = ls[hh]; }
        }
        sync();
        // this rank's partial: merge the warps (fixed order)
        float* st = s.u.w.stage;
        for (int idx = tid; idx < GQ * HD; idx += 256) {
            const int hh = idx / HD, d = idx - hh * HD;
            float ma = -INFINITY;
            for (int w = 0; w < NCW; ++w) ma = fmaxf(ma, s.u.w.wacc[w * PATT + hh * 132 + HD]);
            float a = 0.f, l = 0.f;
            for (int w = 0; w < NCW; ++w) {
                const float* pw = s.u.w.wacc + w * PATT + hh * 132;
                const float c = ma == -INFINITY ? 0.f : expf(pw[HD] - ma);
                a += pw[d] * c;
                l += pw[HD + 1] * c;
            }
            st[hh * 132 + d] = a;
            if (d == 0) { st[hh * 132 + HD] = ma; st[hh * 132 + HD + 1] = l; st[hh * 132 + HD + 2] = 0.f; st[hh * 132 + HD + 3] = 0.f; }
        }
        sync();
        ag_send(st, 1, PATT, s.patt, 0, &s.bar_patt, (unsigned)(CS * PATT * 4));
        ag_wait(&s.bar_patt, n_patt);
        // merge the ranks in order
        for (int idx = tid; idx < GQ * HD; idx += 256) {
            const int hh = idx / HD, d = idx - hh * HD;
            float ma = -INFINITY;
            for (int r = 0; r < CS; ++r) ma = fmaxf(ma, s.patt[r * PATT + hh * 132 + HD]);
            float num = 0.f, den = 0.f;
            for (int r = 0; r < CS; ++r) {
                const float* pr = s.patt + r * PATT + hh * 132;
                const float c = pr[HD] == -INFINITY ? 0.f : expf(pr[HD] - ma);
                num += pr[d] * c;
                den += pr[HD + 1] * c;
            }
            s.u.w.o[idx] = num / den;
        }
        sync();
    }

    __device__ __forceinline__ void op_att(const Op& o) {
        const int M = tokens(o);
        const int p0 = o.talker ? pos : (o.s == 0 ? 0 : o.s + 1);
        att_prep(o, M, p0);
        if (o.talker) att_talker(o);
        else att_pred(o, M, p0);
    }

    // logits words of a head: this CTA's rows (staged), then every reader polls them
    __device__ __forceinline__ void head_rows(int R, Word* dst, unsigned e) {
        for (int t = threadIdx.x; t < R; t += 256) st_word(dst + (size_t)cta * R + t, s.u.w.stage[t], e);
    }
    // poll n logit words into l[]
    __device__ __forceinline__ void fetch_logits(const Word* src, int n, unsigned e, float* l) {
        for (int i = threadIdx.x; i < n; i += 4 * 256) {
            const Word* p[4];
            Word w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) p[j] = src + min(i + 256 * j, n - 1);
            poll<4>(w, p, e);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (i + 256 * j < n) l[i + 256 * j] = val_of(w[j]);
        }
    }

    // predictor head rows are staged: publish them, gather all logits, draw (every CTA)
    __device__ __forceinline__ void headc_tail(const Op& o, int R) {
        const unsigned e = next_epoch();
        Word* lg = P.lg + (size_t)(head_cnt++ & 1) * P.cpV;
        head_rows(R, lg, e);
        // the draw's scratch overlays the Work buffers: every warp is past them
        sync();
        auto& sm = s.u.draw;
        fetch_logits(lg, P.cpV, e, sm.l);
        sync();
        if (cta == 0 && P.cap_c && P.cap_slot[0] >= 0 && frame < P.cap_T) {
            float* dst = P.cap_c + (((size_t)P.cap_slot[0] * P.cap_T + frame) * (P.G - 1) + o.s) * P.cpV;
            for (int i = threadIdx.x; i < P.cpV; i += 256) dst[i] = sm.l[i];
        }
        const q3tts_sampling p = P.P[0];
        const DrawCfg d{p.cp_do_sample, p.cp_temperature, p.cp_top_k, p.cp_top_p};
        int id = sample_row(sm, nullptr, P.cpV, d, false, 1.0f, nullptr, nullptr, 0, 0, -1, 0, 0, p.seed, 0u,
                            (uint32_t)frame, (uint32_t)(o.s + 1));
        if (fail) id = 0;   // aborting: any in-range id keeps the rest of the walk in bounds
        if (id < 0) {
            // NaN / +inf logits: the row ends with an error (the same on every CTA)
            if (threadIdx.x == 0 && cta == 0) {
                RowState& rs = P.rows[0];
                rs.finished = 1;
                rs.reason = Q3_FINISHED_ERROR;
                rs.frames = frame;
                atomicOr(P.err, ERRB_NAN);
            }
            id = 0;
            fail = true;
        }
        if (threadIdx.x == 0) {
            s.codes[o.s + 1] = id;
            if (cta == 0) P.codes[(size_t)frame * MAX_GROUPS + o.s + 1] = id;
        }
        sync();
    }

    __device__ __forceinline__ void op_tin() {
        // talker input slice: + this step's text row (tts_pad once the text runs out)
        const RowState& rs = P.rows[0];
        const float* tx = frame < rs.n_text ? P.text + (size_t)(rs.text_off + frame) * P.H : P.pad;
        const int Rt = P.H / CS;
        // the last codebook's table row (drawn by the final predictor pass)
        tacc_add_table(P.G - 1);
        for (int i = threadIdx.x; i < Rt; i += 256) s.u.w.stage[i] = s.tacc[i] + __ldcg(tx + rank * Rt + i);
        sync();
        ag_send(s.u.w.stage, 1, Rt, s.x, P.H, &s.bar_x, (unsigned)(P.H * 4));
        ag_wait(&s.bar_x, n_x);
    }

    // talker head rows are staged: publish them; CTA 0 gathers all logits and selects
    __device__ __forceinline__ void headt_tail(int R) {
        const unsigned e = next_epoch();
        Word* lg = P.lg + 2 * (size_t)P.cpV;
        head_rows(R, lg, e);
        if (cta != 0) return;
        // CTA 0 selects: the ring is drained (the head was the last window)
        sync();
        SampSmem& sm = *reinterpret_cast<SampSmem*>(&s.ring[0][0]);
        fetch_logits(lg, P.V, e, sm.l);
        sync();
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
        if (threadIdx.x == 0 && !fail) {
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

    // Every GEMV op (projection, q/k/v, O, gate/up, down, heads) runs through the
    // same code: input, operand, GEMV, epilogue, exchange, each written once, so
    // the loop's instructions stay cached from one op to the next.
    __device__ __forceinline__ void run() {
        const int nops = n_ops(P);
        for (int i = 0; i < nops; ++i) {
            const Op o = op_at(i, P);
            if (o.kind == OP_ATT) { op_att(o); continue; }
            if (o.kind == OP_TIN) { op_tin(); continue; }
            const int M = tokens(o);
            const int H = o.talker ? P.H : P.Hc;
            const int Fc = (o.talker ? P.F : P.Fc) / NCL;
            const bool head = o.kind == OP_HEADC || o.kind == OP_HEADT;
            const int Mg = head ? 1 : M;                 // tokens through this GEMV
            const bool norm = o.kind == OP_QKV || o.kind == OP_GU || head;
            const Gv gv = gemv_of(o, P, cta);
            // ---- input: the predictor pass's token(s) straight into the residual
            if (o.kind == OP_QKV && !o.talker && o.l == 0 && P.H == P.Hc) {
                for (int m = 0; m < M; ++m)
                    for (int k = threadIdx.x; k < H; k += 256) s.x[m * H + k] = token_val(o.s, m, k);
                tacc_add_table(o.s);
                sync();
            }
            // ---- operand
            int sd = -1;
            if (norm) {
                sd = side_take();
                if (o.kind == OP_QKV) qkv_side = sd;
                const float* xsrc = s.x + (o.kind == OP_HEADC ? (M - 1) * H : 0);
                build_norm(xsrc, Mg, H, s.side[sd]);
            } else if (o.kind == OP_PROJ) {
                const int Kp = P.H / NCL;
                for (int m = 0; m < M; ++m)
                    for (int k = threadIdx.x; k < Kp; k += 256) put_op(m, Kp, k, token_val(o.s, m, g * Kp + k));
                tacc_add_table(o.s);
            } else {
                const float* src = o.kind == OP_O ? s.u.w.o : s.a;
                const int ld = o.kind == OP_O ? GQ * HD : Fc;
                build_plain(src, ld, M, gv.K);
            }
            // ---- GEMV
            gemv(gv, Mg);
            if (o.kind == OP_HEADT && cta == 0) {
                // the post-norm hidden feeds the next step's predictor
                const float r = s.u.w.rs[0];
                for (int k = threadIdx.x; k < P.H; k += 256) P.h[k] = s.x[k] * s.side[sd][k] * r;
            }
            if (norm && o.kind != OP_QKV) side_release(sd);
            // ---- epilogue: this CTA's outputs into the stage
            const bool gated = o.kind == OP_GU;
            const int Ro = gated ? gv.R / 2 : gv.R;
            for (int t = threadIdx.x; t < Mg * Ro; t += 256) {
                const int m = t / Ro, k = t - m * Ro;
                float v = gsum(gv, k, m, Mg);
                if (norm) v *= s.u.w.rs[m];
                if (gated) {
                    const float up = gsum(gv, Ro + k, m, Mg) * s.u.w.rs[m];
                    v = v / (1.0f + expf(-v)) * up;
                }
                s.u.w.stage[t] = v;
            }
            // ---- exchange
            if (o.kind == OP_QKV || o.kind == OP_GU) {
                sync();
                const bool q = o.kind == OP_QKV;
                ag_send(s.u.w.stage, M, Ro, q ? s.qkv : s.a, q ? QKVR : Fc, q ? &s.bar_qkv : &s.bar_a,
                        (unsigned)(M * (q ? QKVR : Fc) * 4));
                ag_wait(q ? &s.bar_qkv : &s.bar_a, q ? n_qkv : n_a);
            } else if (o.kind == OP_HEADC) {
                headc_tail(o, gv.R);
            } else if (o.kind == OP_HEADT) {
                headt_tail(gv.R);
            } else {
                reduce_x(M, gv.R, H, o.kind != OP_PROJ, o.kind == OP_PROJ ? P.cp_proj_b : nullptr);
            }
        }
    }
};

__global__ void __launch_bounds__(NT, 1) cluster_step_kernel(const ClParams* __restrict__ Pp) {
    extern __shared__ __align__(128) unsigned char smraw[];
    __shared__ __align__(16) ClParams sP;   // the launch's parameters, read from shared memory
    Sm& s = *reinterpret_cast<Sm*>(smraw);
    for (int i = threadIdx.x; i < (int)(sizeof(ClParams) / 4); i += NT)
        reinterpret_cast<uint32_t*>(&sP)[i] = reinterpret_cast<const uint32_t*>(Pp)[i];
    __syncthreads();
    const ClParams& P = sP;
    const RowState& rs0 = P.rows[0];
    if (rs0.finished || aborted(P)) return;   // uniform over the grid
    const int frame = rs0.sel - 1, pos = rs0.pos, code0 = rs0.code0;
    if (frame < 0 || frame >= P.frames_cap || code0 < 0 || code0 >= P.V || rs0.sel >= (1 << 21) || pos < 1 ||
        pos >= P.cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(P.err, ERRB_BOUNDS);
        return;
    }
    // the exchanges address peer CTAs by cluster rank: anything but 8 clusters of
    // 8 CTAs (e.g. a launch without its cluster shape) returns before any of them
    if (gridDim.x != NCTA || cl_nctarank() != CS || cl_nclusters() != NCL) {
        if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(P.err, ERRB_LAUNCH);
        return;
    }
    const int cta = (int)blockIdx.x, g = (int)cl_id(), rank = (int)cl_rank();
    if (threadIdx.x == 0) {
        for (int i = 0; i < NSLOT; ++i) { mbar_init(&s.full[i], 1); mbar_init(&s.empty[i], NCW); }
        mbar_init(&s.bar_qkv, 1);
        mbar_init(&s.bar_x, 1);
        mbar_init(&s.bar_a, 1);
        mbar_init(&s.bar_patt, 1);
        for (int i = 0; i < 2; ++i) { mbar_init(&s.side_full[i], 1); mbar_init(&s.side_empty[i], NCW); }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s.codes[0] = code0;
        if (cta == 0) P.codes[(size_t)frame * MAX_GROUPS] = code0;
    }
    // talker input slice starts with codec_emb(code0)
    {
        const int Rt = P.H / CS;
        const bf16* ce = (const bf16*)P.codec_emb + (size_t)code0 * P.H + rank * Rt;
        for (int i = threadIdx.x; i < Rt; i += NT) s.tacc[i] = __bfloat162float(ce[i]);
    }
    // peers write into this CTA's buffers only after every mbarrier is initialised
    cluster_sync_all();
    const int warp = threadIdx.x >> 5;
    if (warp == NCW) {
        if ((threadIdx.x & 31) == 0) {
            Producer pr{s, P, cta, rank, pos};
            pr.run();
            pr.drain();
        }
    } else {
        Consumer c{s, P, cta, g, rank, frame, pos, (unsigned)rs0.sel << 10};
        c.run();
    }
    // no CTA leaves while a peer may still address its shared memory
    cluster_sync_all();
}

// ------------------------------------------------------------------ packing
// dst: NCTA slices of R x K bf16, each in fragment order (16-row blocks, K steps
// of 16, 32 lanes x 16 bytes).  kind: 0 q/k/v, 1 O, 2 gate/up, 3 down, 4 head,
// 5 projection.
__global__ void pack_kernel(const bf16* __restrict__ src, long ld, int kind, int R, int K, int nq, int Fc, int F,
                            int colw, bf16* __restrict__ dst) {
    const long per = (long)R * K / 8;   // 16-byte chunks per CTA slice
    const long n = per * NCTA;
    for (long o = (long)blockIdx.x * blockDim.x + threadIdx.x; o < n; o += (long)gridDim.x * blockDim.x) {
        const int c = (int)(o / per);
        const long rem = o - (long)c * per;
        const int g = c / CS, r = c - g * CS;
        const int nks = K / 16;
        const int b = (int)(rem / ((long)nks * 32));
        const int t = (int)((rem / 32) % nks);
        const int lane = (int)(rem & 31);
        const int gq = lane >> 2, q = lane & 3;
        long row[2];
        for (int h = 0; h < 2; ++h) {
            const int i = 16 * b + gq + 8 * h;
            long rr;
            switch (kind) {
                case 0: {
                    const int j = r * R + i;
                    if (j < GQ * HD) rr = (long)GQ * HD * g + j;
                    else if (j < (GQ + 1) * HD) rr = (long)nq * HD + (long)g * HD + (j - GQ * HD);
                    else rr = (long)nq * HD + (long)NCL * HD + (long)g * HD + (j - (GQ + 1) * HD);
                    break;
                }
                case 2: {
                    const int hr = R / 2;
                    rr = i < hr ? (long)g * Fc + (long)r * hr + i : (long)F + (long)g * Fc + (long)r * hr + (i - hr);
                    break;
                }
                case 4: rr = (long)c * R + i; break;
                default: rr = (long)r * R + i; break;   // O, down, projection: row slice r
            }
            row[h] = rr;
        }
        long col = 0;
        if (kind == 1) col = (long)g * GQ * HD;
        else if (kind == 3) col = (long)g * Fc;
        else if (kind == 5) col = (long)g * colw;
        const long k = col + 16 * t + 2 * q;
        const bf16* a = src + row[0] * ld;
        const bf16* bb = src + row[1] * ld;
        __align__(16) bf16 v[8] = {a[k], a[k + 1], bb[k], bb[k + 1], a[k + 8], a[k + 9], bb[k + 8], bb[k + 9]};
        reinterpret_cast<uint4*>(dst)[o] = *reinterpret_cast<const uint4*>(v);
    }
}

cudaError_t pack_one(const void* src, long ld, int kind, int R, int K, int nq, int Fc, int F, int colw,
                     unsigned char* dst, cudaStream_t st) {
    pack_kernel<<<1216, 256, 0, st>>>((const bf16*)src, ld, kind, R, K, nq, Fc, F, colw, (bf16*)dst);
    return cudaGetLastError();
}

}  // namespace

const char* cl_unsupported(const q3tts_config& c) {
    if (c.dtype != Q3_BF16) return "bf16 only";
    if (c.head_dim != HD || c.n_kv_heads != NCL || c.n_q_heads != GQ * NCL) return "16 q / 8 kv heads of 128";
    if (c.cp_layers > CL_MAX_CP_LAYERS) return "too many predictor layers";
    if (c.n_groups < 2 || c.n_groups > PKV) return "codebooks";
    const int H = c.hidden, Hc = c.cp_hidden;
    if (H % (CS * 16) || Hc % (CS * 16) || H > 2048 || Hc > 1024) return "widths";
    if (H != Hc && (H % (NCL * 16) || H / NCL > 256 * 2)) return "projection width";
    for (int F : {c.ffn, c.cp_ffn}) {
        if (F % (NCL * CS * 8) || (F / NCL / CS) % 8 || 2 * (F / NCL / CS) > 192) return "ffn width";
        if ((F / NCL / CS * 2) % 16) return "ffn width";
    }
    if (c.ffn / NCL > AMAX || 2 * (c.cp_ffn / NCL) > AMAX) return "ffn slice";
    if (c.codec_vocab % (NCTA * 16) || c.cp_vocab % (NCTA * 16) || c.cp_vocab > CPV_MAX) return "vocabularies";
    if (H / CS > TACC) return "talker slice";
    // K-split partial sums of every GEMV fit the CTA's buffer
    auto part = [](int R, int K, int M) {
        const int nb = R / 16, bb = K / 16 * 512;
        const int S = bb <= SLOT ? std::max(1, NCW / std::min(std::min(nb, SLOT / bb), NCW)) : NCW;
        return nb * S * 16 * M;
    };
    const int Fct = c.ffn / NCL, Fcc = c.cp_ffn / NCL;
    const int need[] = {part(QKVR / CS, H, 1), part(H / CS, GQ * HD, 1), part(2 * Fct / CS, H, 1),
                        part(H / CS, Fct, 1), part(QKVR / CS, Hc, 2), part(Hc / CS, GQ * HD, 2),
                        part(2 * Fcc / CS, Hc, 2), part(Hc / CS, Fcc, 2), part(c.cp_vocab / NCTA, Hc, 1),
                        part(c.codec_vocab / NCTA, H, 1), H != Hc ? part(Hc / CS, H / NCL, 2) : 0};
    for (int n : need)
        if (n > PARTN) return "partial sums";
    if (2 * (Hc / CS) > STG || H / CS > STG || 2 * (2 * Fcc / CS) > STG) return "staged outputs";
    if (c.max_ctx > (1 << 20)) return "context";
    return "";
}

ClLayout cl_layout(const q3tts_config& c) {
    ClLayout L{};
    const size_t e = 2;
    const int nqkv = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
    size_t off = 0;
    auto stack = [&](size_t* offs, size_t* pers, int Lr, int H, int F) {
        const size_t sz[4] = {(size_t)nqkv * H * e, (size_t)H * c.n_q_heads * c.head_dim * e, (size_t)2 * F * H * e,
                              (size_t)H * F * e};
        for (int k = 0; k < 4; ++k) {
            offs[k] = off;
            pers[k] = sz[k];
            off += sz[k] * Lr;
        }
    };
    stack(L.off_t, L.per_t, c.n_layers, c.hidden, c.ffn);
    stack(L.off_c, L.per_c, c.cp_layers, c.cp_hidden, c.cp_ffn);
    L.off_cph = off;
    L.per_cph = (size_t)c.cp_vocab * c.cp_hidden * e;
    off += L.per_cph * (c.n_groups - 1);
    L.off_th = off;
    off += (size_t)c.codec_vocab * c.hidden * e;
    L.off_proj = off;
    if (c.hidden != c.cp_hidden) off += (size_t)c.cp_hidden * c.hidden * e;
    L.pack_bytes = off;
    L.xr_words = (size_t)2 * NCL * 2 * XW;
    L.lg_words = (size_t)2 * c.cp_vocab + c.codec_vocab;
    return L;
}

static_assert(sizeof(SampSmem) <= sizeof(Sm::ring), "talker draw scratch must fit the drained ring");
static_assert(sizeof(Sm) + sizeof(ClParams) <= 227 * 1024, "shared memory of one CTA");
static_assert(sizeof(ClParams) % 4 == 0, "parameters are copied in 32-bit words");

size_t cl_smem_bytes() { return sizeof(Sm); }

cudaError_t cl_setup() {
    cudaError_t e = cudaFuncSetAttribute(cluster_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(Sm));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(NCTA);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = sizeof(Sm);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int ncl = 0;
    e = cudaOccupancyMaxActiveClusters(&ncl, cluster_step_kernel, &cfg);
    if (e != cudaSuccess) return e;
    return ncl >= NCL ? cudaSuccess : cudaErrorCooperativeLaunchTooLarge;
}

cudaError_t cl_pack_weights(const q3tts_config& c, const q3tts_weights& w, unsigned char* pack, cudaStream_t st) {
    const ClLayout L = cl_layout(c);
    const int nq = c.n_q_heads;
    const int nqkv = (nq + 2 * c.n_kv_heads) * HD;
    auto stack = [&](const q3tts_block_weights& b, const size_t* offs, const size_t* pers, int Lr, int H,
                     int F) -> cudaError_t {
        const int Fc = F / NCL;
        for (int l = 0; l < Lr; ++l) {
            cudaError_t e;
            e = pack_one((const char*)b.wqkv + (size_t)l * nqkv * H * 2, H, 0, QKVR / CS, H, nq, Fc, F, 0,
                         pack + offs[0] + l * pers[0], st);
            if (e != cudaSuccess) return e;
            e = pack_one((const char*)b.wo + (size_t)l * H * nq * HD * 2, nq * HD, 1, H / CS, GQ * HD, nq, Fc, F, 0,
                         pack + offs[1] + l * pers[1], st);
            if (e != cudaSuccess) return e;
            e = pack_one((const char*)b.wgu + (size_t)l * 2 * F * H * 2, H, 2, 2 * Fc / CS, H, nq, Fc, F, 0,
                         pack + offs[2] + l * pers[2], st);
            if (e != cudaSuccess) return e;
            e = pack_one((const char*)b.wd + (size_t)l * H * F * 2, F, 3, H / CS, Fc, nq, Fc, F, 0,
                         pack + offs[3] + l * pers[3], st);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    };
    cudaError_t e = stack(w.talker, L.off_t, L.per_t, c.n_layers, c.hidden, c.ffn);
    if (e != cudaSuccess) return e;
    e = stack(w.cp, L.off_c, L.per_c, c.cp_layers, c.cp_hidden, c.cp_ffn);
    if (e != cudaSuccess) return e;
    for (int s = 0; s < c.n_groups - 1; ++s) {
        e = pack_one((const char*)w.cp_heads + (size_t)s * c.cp_vocab * c.cp_hidden * 2, c.cp_hidden, 4,
                     c.cp_vocab / NCTA, c.cp_hidden, nq, 0, 0, 0, pack + L.off_cph + s * L.per_cph, st);
        if (e != cudaSuccess) return e;
    }
    e = pack_one(w.codec_head, c.hidden, 4, c.codec_vocab / NCTA, c.hidden, nq, 0, 0, 0, pack + L.off_th, st);
    if (e != cudaSuccess) return e;
    if (c.hidden != c.cp_hidden)
        e = pack_one(w.cp_proj_w, c.hidden, 5, c.cp_hidden / CS, c.hidden / NCL, nq, 0, 0, c.hidden / NCL,
                     pack + L.off_proj, st);
    return e;
}

cudaError_t launch_cluster_step(const ClParams* params_dev, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(NCTA);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = sizeof(Sm);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, cluster_step_kernel, params_dev);
}

}  // namespace q3
