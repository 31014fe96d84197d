// Tensor-core projections for many tokens at once (large batches, prefill
// chunks): Y[m][n] (+)= sum_k W[n][k] X[m][k], bf16 weights, fp32 inputs and
// accumulation.  The fp32 input is split exactly enough into two bf16 parts
// (x = hi + lo + O(2^-18 |x|)) and both parts go through the tensor cores.
//
// The weight matrix is the MMA's A operand (128 weight rows per tile) and the
// tokens are its N dimension (NT tokens per tile), so D[n][m] = W_tile . X^T
// lives in tensor memory as 128 lanes (weight rows) x NT fp32 columns.
//   - TMA (cp.async.bulk.tensor, 128-byte swizzle) stages 64-wide K slices of
//     both operands into a shared-memory ring as deep as ~192 KB allows
//     (mbarrier completion);
//   - one thread issues tcgen05.mma (kind::f16, M=128, N=NT, K=16 per
//     instruction; W x hi, then W x lo into the same accumulator) and commits
//     each stage back to the producer;
//   - after the last stage, the four warps read their 32 TMEM lanes with
//     tcgen05.ld and apply the epilogue (store / residual add / bias, or
//     SiLU(g)*u for the stacked gate/up weights, which uses two accumulators).
//   - when the output tiles alone cannot fill the GPU, K is split over the
//     CTAs of a thread-block cluster (one output tile per cluster).  Once every
//     CTA of the cluster has drained its operand ring (cluster barrier), each
//     pushes its fp32 accumulator, column share by column share, into the ring
//     of the CTA that owns those columns (distributed shared memory, vector
//     stores); after a second barrier CTA z sums the z-th share over the splits
//     in split order and applies the epilogue.
// Every mbarrier wait is bounded; an expired wait sets the timeout error bit,
// the CTA skips its remaining work, frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "pdl.cuh"

#include <algorithm>

namespace q3 {

namespace {

constexpr int BM = 128;        // weight rows per tile (MMA M)
constexpr int BK = 64;         // K per stage (one 128-byte swizzle row of bf16)
constexpr int RING_BYTES = 192 * 1024;
// ring depth for a tile shape: stages of (BM (x2 gated) + 2 NT) x BK bf16
constexpr int stages_for(int nt, bool gated) {
    const int st = RING_BYTES / ((BM * (gated ? 2 : 1) + 2 * nt) * BK * 2);
    return st > 8 ? 8 : st;
}
constexpr long long TC_WAIT_LIMIT = 2000000000LL;

__device__ __forceinline__ uint32_t s_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mb_init(uint64_t* b, unsigned n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(s_u32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mb_expect_tx(uint64_t* b, unsigned bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
                 ::"r"(s_u32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mb_try(uint64_t* b, unsigned parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(s_u32(b)), "r"(parity) : "memory");
    return ok != 0;
}
__device__ bool mb_wait(uint64_t* b, unsigned parity, int* err) {
    if (mb_try(b, parity)) return true;
    const long long t0 = clock64();
    while (!mb_try(b, parity))
        if (clock64() - t0 > TC_WAIT_LIMIT) {
            atomicOr(err, ERRB_TIMEOUT);
            return false;
        }
    return true;
}
__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(s_u32(dst)), "l"((uint64_t)map), "r"(x), "r"(y), "r"(s_u32(bar)) : "memory");
}

// Shared-memory matrix descriptor: K-major tile with 128-byte swizzle, rows of
// 128 bytes, 8-row core groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);       // start address
    d |= (uint64_t)1 << 16;                          // leading byte offset (unused for this layout)
    d |= (uint64_t)(1024 >> 4) << 32;                // stride byte offset
    d |= (uint64_t)1 << 46;                          // descriptor version
    d |= (uint64_t)2 << 61;                          // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: fp32 D, bf16 A and B, both K-major.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, int acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(s_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// address of shared location a in cluster CTA `rank`
__device__ __forceinline__ uint32_t map_peer(uint32_t a, int rank) {
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    return ra;
}
// four fp32 to a peer's shared memory (address from map_peer)
__device__ __forceinline__ void st_dsmem4(uint32_t ra, float a, float b, float c, float d) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(ra), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

template <int NT, bool GATED, int STAGES>
struct TcSmem {
    alignas(1024) bf16 a[STAGES][BM * BK];
    alignas(1024) bf16 a2[GATED ? STAGES : 1][GATED ? BM * BK : 8];
    alignas(1024) bf16 b[STAGES][NT * BK];
    alignas(1024) bf16 b2[STAGES][NT * BK];
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t done;
    uint32_t tmem;
};

template <int NT>
constexpr uint32_t tmem_cols(bool gated) {
    const int need = gated ? 2 * NT : NT;
    return need <= 32 ? 32 : need <= 64 ? 64 : need <= 128 ? 128 : need <= 256 ? 256 : 512;
}

template <int NT, bool GATED, int STAGES>
__global__ void __launch_bounds__(128, 1) umma_linear_kernel(const __grid_constant__ CUtensorMap tmW,
                                                             const __grid_constant__ CUtensorMap tmX,
                                                             const __grid_constant__ CUtensorMap tmX2, int N, int K,
                                                             int M, float* __restrict__ Y, int ldy,
                                                             const float* __restrict__ bias, int accumulate, int F,
                                                             float* __restrict__ Gout, int ldg, bf16* __restrict__ Ghi,
                                                             bf16* __restrict__ Glo, int kbs, int* err) {
    extern __shared__ __align__(1024) unsigned char raw[];
    // 1024-byte alignment of the swizzled tiles
    unsigned char* base = (unsigned char*)(((uintptr_t)raw + 1023) & ~(uintptr_t)1023);
    TcSmem<NT, GATED, STAGES>& s = *reinterpret_cast<TcSmem<NT, GATED, STAGES>*>(base);
    constexpr uint32_t COLS = tmem_cols<NT>(GATED);
    constexpr uint32_t IDESC = make_idesc(BM, NT);
    constexpr int H2 = GATED ? 2 : 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // grid (ks, weight-row tiles, token tiles); cluster (ks, 1, 1): rank = K split
    const int n0 = blockIdx.y * BM, m0 = blockIdx.z * NT;
    const int ks = gridDim.x, kz = blockIdx.x;
    // this CTA's K blocks [kb0, kb0 + nk)
    const int nk_all = (K + BK - 1) / BK;
    const int kb0 = kz * kbs;
    const int nk = min(kbs, nk_all - kb0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) { mb_init(&s.full[i], 1); mb_init(&s.empty[i], 1); }
        mb_init(&s.done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(s_u32(&s.tmem)),
                     "r"(COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem;
    bool ok = true;
    int issued = 0, committed = 0;   // stages the producer issued / the MMA issuer committed
    // Programmatic dependent launch: this grid touches nothing the previous
    // kernel writes before griddepcontrol.wait returns (the previous grid
    // complete, its writes visible); only the weights, which no kernel
    // writes, are read before that.  The next launch may start once every CTA
    // of this grid has finished its main loop (below).

    if (warp == 0 && lane == 0) {
        // producer: K slices of W (and of the up half) and of X; the first
        // ring's worth of W is requested before the previous kernel is done
        const unsigned bytes = (unsigned)((BM * (GATED ? 2 : 1) + 2 * NT) * BK * sizeof(bf16));
        const int pre = min(nk, STAGES);
        issued = pre;
        for (int kb = 0; kb < pre; ++kb) {
            mb_expect_tx(&s.full[kb], bytes);
            const int kx = (kb0 + kb) * BK;
            tma_2d(s.a[kb], &tmW, kx, n0, &s.full[kb]);
            if (GATED) tma_2d(s.a2[kb], &tmW, kx, F + n0, &s.full[kb]);
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        for (int kb = 0; kb < pre; ++kb) {
            const int kx = (kb0 + kb) * BK;
            tma_2d(s.b[kb], &tmX, kx, m0, &s.full[kb]);
            tma_2d(s.b2[kb], &tmX2, kx, m0, &s.full[kb]);
        }
        for (int kb = pre; kb < nk && ok; ++kb) {
            const int st = kb % STAGES;
            const unsigned round = kb / STAGES;
            if (!mb_wait(&s.empty[st], (round - 1) & 1, err)) { ok = false; break; }
            mb_expect_tx(&s.full[st], bytes);
            const int kx = (kb0 + kb) * BK;
            tma_2d(s.a[st], &tmW, kx, n0, &s.full[st]);
            if (GATED) tma_2d(s.a2[st], &tmW, kx, F + n0, &s.full[st]);
            tma_2d(s.b[st], &tmX, kx, m0, &s.full[st]);
            tma_2d(s.b2[st], &tmX2, kx, m0, &s.full[st]);
            issued = kb + 1;
        }
    } else {
        // everyone else starts its bounded waits only once the previous grid is done
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }
    if (warp == 1 && lane == 0) {
        // MMA issuer
        for (int kb = 0; kb < nk && ok; ++kb) {
            const int st = kb % STAGES;
            if (!mb_wait(&s.full[st], (kb / STAGES) & 1, err)) { ok = false; break; }
            tc_fence_after();
            const uint64_t da = sw128_desc(s_u32(s.a[st]));
            const uint64_t db = sw128_desc(s_u32(s.b[st]));
            const uint64_t db2 = sw128_desc(s_u32(s.b2[st]));
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
                // advance 16 bf16 (32 bytes) along K inside the swizzled row
                umma(tmem, da + 2 * kk, db + 2 * kk, IDESC, (kb | kk) != 0);
                umma(tmem, da + 2 * kk, db2 + 2 * kk, IDESC, 1);
                if (GATED) {
                    const uint64_t da2 = sw128_desc(s_u32(s.a2[st]));
                    umma(tmem + NT, da2 + 2 * kk, db + 2 * kk, IDESC, (kb | kk) != 0);
                    umma(tmem + NT, da2 + 2 * kk, db2 + 2 * kk, IDESC, 1);
                }
            }
            umma_commit(&s.empty[st]);
            committed = kb + 1;
        }
        if (ok) umma_commit(&s.done);
    }
    __syncwarp();
    // epilogue: warp w owns TMEM lanes 32w..32w+31 (weight rows n0+32w..)
    const bool have = __all_sync(0xffffffffu, mb_wait(&s.done, 0, err));
    // the operand stream is done: the next kernel may set up and request its weights
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    tc_fence_after();
    const int row = warp * 32 + lane;
    const int n = n0 + row;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    // final values of this thread's row for tokens m0 + c0 .. c0 + 15
    auto finish = [&](int c0, const float (&v)[16], const float (&u)[16]) {
        if (GATED) {
            if (n < F) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int m = m0 + c0 + j;
                    if (m < M) {
                        const float a = v[j] / (1.0f + expf(-v[j])) * u[j];
                        if (Ghi) {
                            // the next projection's tensor-core operand, [M][F] bf16 high / low
                            const bf16 h = __float2bfloat16_rn(a);
                            Ghi[(size_t)m * F + n] = h;
                            Glo[(size_t)m * F + n] = __float2bfloat16_rn(a - __bfloat162float(h));
                        } else {
                            Gout[(size_t)m * ldg + n] = a;
                        }
                    }
                }
            }
        } else if (n < N) {
            const float bn = bias ? bias[n] : 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int m = m0 + c0 + j;
                if (m < M) {
                    float* y = Y + (size_t)m * ldy + n;
                    *y = accumulate ? *y + v[j] + bn : v[j] + bn;
                }
            }
        }
    };
    // Plain outputs go through the drained ring as a [NT][BM] fp32 tile: the
    // residual (accumulate) comes in and the result goes out with coalesced
    // 16-byte accesses, every load in flight at once, instead of one L2 round
    // trip per 16 columns of each thread's row.
    bool staged = false;
    if constexpr (!GATED) {
        const bool fits = ks == 1 && ldy % 4 == 0 && ((uintptr_t)Y & 15) == 0;
        staged = __syncthreads_and(have && fits) != 0;
    }
    if (staged) {
        float* tile = reinterpret_cast<float*>(s.a);   // [NT][BM], ring drained
        const int mrows = min(NT, M - m0), ncols = min(BM, N - n0);
        constexpr int C4 = BM / 4;
        if (accumulate) {
            for (int i = threadIdx.x; i < NT * C4; i += 128) {
                const int m = i / C4, c = (i - m * C4) * 4;
                if (m >= mrows) continue;
                const float* src = Y + (size_t)(m0 + m) * ldy + n0 + c;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (c + 3 < ncols) {
                    v = *reinterpret_cast<const float4*>(src);
                } else {
                    if (c < ncols) v.x = src[0];
                    if (c + 1 < ncols) v.y = src[1];
                    if (c + 2 < ncols) v.z = src[2];
                }
                *reinterpret_cast<float4*>(tile + m * BM + c) = v;
            }
            __syncthreads();
        }
        const float bn = (bias && n < N) ? bias[n] : 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < NT; c0 += 16) {
            float v[16];
            tmem_ld16(lane_base + c0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                float* t = tile + (c0 + j) * BM + row;
                *t = accumulate ? *t + v[j] + bn : v[j] + bn;
            }
        }
        __syncthreads();
        for (int i = threadIdx.x; i < NT * C4; i += 128) {
            const int m = i / C4, c = (i - m * C4) * 4;
            if (m >= mrows) continue;
            float* dst = Y + (size_t)(m0 + m) * ldy + n0 + c;
            const float4 v = *reinterpret_cast<const float4*>(tile + m * BM + c);
            if (c + 3 < ncols) {
                *reinterpret_cast<float4*>(dst) = v;
            } else {
                if (c < ncols) dst[0] = v.x;
                if (c + 1 < ncols) dst[1] = v.y;
                if (c + 2 < ncols) dst[2] = v.z;
            }
        }
    } else if (ks == 1) {
        if (have) {
#pragma unroll 1
            for (int c0 = 0; c0 < NT; c0 += 16) {
                float v[16], u[16];
                tmem_ld16(lane_base + c0, v);
                if (GATED) tmem_ld16(lane_base + NT + c0, u);
                finish(c0, v, u);
            }
        }
    } else {
        // owner z of token columns [z per, z per + per) keeps an inbox in its
        // drained ring: [split][H2][row][per + 4] fp32 (padded rows)
        const int per = (NT / 16 + ks - 1) / ks * 16;
        const int rs = per + 4;
        const uint32_t inbox = s_u32(s.a);
        cluster_sync();   // every ring of the cluster is drained
        if (have) {
#pragma unroll 1
            for (int c0 = 0; c0 < NT; c0 += 16) {
                const int o = c0 / per, cl = c0 - o * per;
                float v[16], u[16];
                tmem_ld16(lane_base + c0, v);
                if (GATED) tmem_ld16(lane_base + NT + c0, u);
#pragma unroll
                for (int h = 0; h < H2; ++h) {
                    const float* src = h ? u : v;
                    const uint32_t dst =
                        map_peer(inbox + (uint32_t)((((kz * H2 + h) * BM + row) * rs + cl) * 4), o);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        st_dsmem4(dst + 16u * q, src[4 * q], src[4 * q + 1], src[4 * q + 2], src[4 * q + 3]);
                }
            }
        }
        cluster_sync();   // every push has landed
        const float* box = reinterpret_cast<const float*>(s.a);
#pragma unroll 1
        for (int cl = 0; cl < per && kz * per + cl < NT; cl += 16) {
            float v[16], u[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) { v[j] = 0.f; u[j] = 0.f; }
            for (int z = 0; z < ks; ++z) {
#pragma unroll
                for (int h = 0; h < H2; ++h) {
                    const float4* q = reinterpret_cast<const float4*>(box + ((z * H2 + h) * BM + row) * rs + cl);
                    float* d = h ? u : v;
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        const float4 f = q[k4];
                        d[4 * k4] += f.x; d[4 * k4 + 1] += f.y; d[4 * k4 + 2] += f.z; d[4 * k4 + 3] += f.w;
                    }
                }
            }
            finish(kz * per + cl, v, u);
        }
    }
    if (!have) {
        // a wait ran out: nothing may still be writing this CTA's shared memory
        // or tensor memory when it leaves (bounded waits for the copies the
        // producer issued and for the MMAs behind the last commit)
        if (warp == 0 && lane == 0)
            for (int kb = max(0, issued - STAGES); kb < issued; ++kb)
                mb_wait(&s.full[kb % STAGES], (kb / STAGES) & 1, err);
        if (warp == 1 && lane == 0 && committed > 0)
            mb_wait(&s.empty[(committed - 1) % STAGES], ((committed - 1) / STAGES) & 1, err);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(COLS) : "memory");
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// 2-D bf16 map over [rows][cols] (row stride ld elements), box [box_rows][64].
bool make_map(CUtensorMap* m, const void* base, int rows, int cols, int ld, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * sizeof(bf16)};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// x -> (hi, lo): hi = bf16(x), lo = bf16(x - hi); [M][K] each, row stride K.
// Grid (ceil(K / 1024), M): each thread converts 4 consecutive elements
// (K and ldx are multiples of 8, so the float4 reads are aligned).
__global__ void split_kernel(const float* __restrict__ X, int ldx, int M, int K, bf16* __restrict__ hi,
                             bf16* __restrict__ lo) {
    pdl_wait();
    pdl_trigger();
    const int m = blockIdx.y;
    const int k = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (m >= M || k >= K) return;
    const float4 x = *reinterpret_cast<const float4*>(X + (size_t)m * ldx + k);
    const float xs[4] = {x.x, x.y, x.z, x.w};
    __align__(8) bf16 h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        h[i] = __float2bfloat16_rn(xs[i]);
        l[i] = __float2bfloat16_rn(xs[i] - __bfloat162float(h[i]));
    }
    *reinterpret_cast<uint2*>(hi + (size_t)m * K + k) = *reinterpret_cast<const uint2*>(h);
    *reinterpret_cast<uint2*>(lo + (size_t)m * K + k) = *reinterpret_cast<const uint2*>(l);
}

// Clusters of `ks` CTAs of this kernel that can be resident at once (cached).
template <int NT, bool GATED>
int cluster_capacity(int ks) {
    constexpr int STAGES = stages_for(NT, GATED);
    static int cap[9] = {0};
    if (ks < 1 || ks > 8) return 0;
    if (cap[ks] == 0) {
        const size_t smem = sizeof(TcSmem<NT, GATED, STAGES>) + 1024;
        if (cudaFuncSetAttribute(umma_linear_kernel<NT, GATED, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(ks, 1, 1);
        cfg.blockDim = dim3(128);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = ks;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, (void*)umma_linear_kernel<NT, GATED, STAGES>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = ks == 1 ? device_sm_count() : 0;
        }
        cap[ks] = n > 0 ? n : -1;
    }
    return cap[ks] > 0 ? cap[ks] : 0;
}

// Resident CTAs of this kernel at once (1 CTA per SM: ~192 KB of shared memory).
template <int NT, bool GATED>
int resident_ctas(int ks) {
    return ks == 1 ? device_sm_count() : cluster_capacity<NT, GATED>(ks) * ks;
}

// Time (microseconds) of an NT-wide tile shape split ks ways, a model fitted
// to CUDA-event timings of this kernel on the GB300 over the projection shapes
// of the frame loop and the prefill (M = 16..8192 tokens, N = 1024..6144
// rows, K = 1024..6144; every tile width and split): each CTA streams its
// operands at about 80 GB/s (its ring in flight), a wave costs 0.5 us more,
// and a split's reduction pushes the fp32 accumulator through distributed
// shared memory at about 20 GB/s per CTA.  Clusters of 2 / 4 / 8 CTAs keep at
// most 136 / 112 / 96 CTAs busy (fewer if the occupancy query says so).
// Over the calibration set this picks within 2 % of the best shape on
// average (worst 17 %).  Returns the best ks and its cost.
template <int NT, bool GATED>
double best_split(int nrows, int M, int K, int* ks_out) {
    constexpr int H2 = GATED ? 2 : 1;
    constexpr size_t stage = (size_t)(BM * H2 + 2 * NT) * BK * sizeof(bf16);
    constexpr size_t ring = (size_t)stages_for(NT, GATED) * stage;
    constexpr double per_wave_us = 0.5, stream_bytes_per_us = 80e3, reduce_bytes_per_us = 20e3;
    const int tiles = ((nrows + BM - 1) / BM) * ((M + NT - 1) / NT);
    const int nk = (K + BK - 1) / BK;
    double best = 1e300;
    *ks_out = 1;
    for (int ks : {1, 2, 4, 8}) {
        if (ks > 1 && ks > nk / 2) continue;
        const int per = (NT / 16 + ks - 1) / ks * 16;
        if (ks > 1 && (size_t)ks * H2 * BM * (per + 4) * sizeof(float) > ring) continue;   // inbox must fit
        int res = resident_ctas<NT, GATED>(ks);
        if (res <= 0) continue;
        if (ks > 1) res = std::min(res, ks == 2 ? 136 : ks == 4 ? 112 : 96);
        const int kbs = (nk + ks - 1) / ks;
        const int waves = (tiles * ks + res - 1) / res;
        double cost = waves * (per_wave_us + kbs * (double)stage / stream_bytes_per_us);
        if (ks > 1) cost += waves * ((double)H2 * BM * NT * sizeof(float) / reduce_bytes_per_us);
        if (cost < best) { best = cost; *ks_out = ks; }
    }
    return best;
}

template <int NT, bool GATED>
cudaError_t launch_tc(const void* W, int N, int K, const float* X, int ldx, int M, float* Y, int ldy,
                      const float* bias, int accumulate, int F, float* G, int ldg, int ks, const TcScratch& tc,
                      int* err, cudaStream_t st, const TcScratch* gsplit = nullptr) {
    constexpr int STAGES = stages_for(NT, GATED);
    bf16* hi = (bf16*)tc.base;
    bf16* lo = hi + (size_t)M * K;
    // X = NULL: the producer of the operand wrote hi / lo itself
    if (X) launch_pdl(split_kernel, dim3((K + 1023) / 1024, M), 256, 0, st, X, ldx, M, K, hi, lo);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CUtensorMap mw, mx, mx2;
    const int wrows = GATED ? 2 * F : N;
    if (!make_map(&mw, W, wrows, K, K, BM) || !make_map(&mx, hi, M, K, K, NT) || !make_map(&mx2, lo, M, K, K, NT))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(TcSmem<NT, GATED, STAGES>) + 1024;
    static bool attr_set = false;
    if (!attr_set) {
        e = cudaFuncSetAttribute(umma_linear_kernel<NT, GATED, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int nrows = GATED ? F : N;
    const int nk = (K + BK - 1) / BK;
    const int kbs = (nk + ks - 1) / ks;
    ks = (nk + kbs - 1) / kbs;   // every split gets at least one K block
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ks, (nrows + BM - 1) / BM, (M + NT - 1) / NT);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // may overlap the previous kernel's tail (the kernel waits for it before
    // reading anything it writes)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    bf16* ghi = nullptr;
    bf16* glo = nullptr;
    if (gsplit) {
        if (!GATED || !tc_fits(*gsplit, M, F)) return cudaErrorInvalidValue;
        ghi = (bf16*)gsplit->base;
        glo = ghi + (size_t)M * F;
    }
    return cudaLaunchKernelEx(&cfg, umma_linear_kernel<NT, GATED, STAGES>, mw, mx, mx2, N, K, M, Y, ldy, bias,
                              accumulate, F, G, ldg, ghi, glo, kbs, err);
}

}  // namespace

#ifdef Q3_GEMM_CALIBRATION
// Calibration builds only (calibrate_gemm.cu times every tile width and split
// the model chooses among): a forced shape, and whether a shape is legal.
int g_force_nt = -1, g_force_ks = 1;
bool tc_shape_ok(int NT, int ks, bool gated, int K);
#endif

namespace {

// Tile width and K split of least cost among the widths the tokens allow.
template <bool GATED>
void pick_shape(int nrows, int M, int K, int* nt, int* ks) {
#ifdef Q3_GEMM_CALIBRATION
    if (g_force_nt > 0) { *nt = g_force_nt; *ks = g_force_ks; return; }
#endif
    double best = 1e300;
    for (int w : {128, 64, 32}) {
        if (w > 32 && w > ((M + 31) / 32) * 32) continue;
        int k = 1;
        const double c = w == 128 ? best_split<128, GATED>(nrows, M, K, &k)
                       : w == 64 ? best_split<64, GATED>(nrows, M, K, &k) : best_split<32, GATED>(nrows, M, K, &k);
        if (c < best) { best = c; *nt = w; *ks = k; }
    }
}

}  // namespace

bool tc_available() { return encode_fn() != nullptr; }

#ifdef Q3_GEMM_CALIBRATION
// the split-K inbox must fit the ring, every split needs two K blocks, and the
// cluster shape must be able to run
bool tc_shape_ok(int NT, int ks, bool gated, int K) {
    const int nk = (K + BK - 1) / BK;
    if (ks > 1 && ks > nk / 2) return false;
    if (ks == 1) return true;
    const int H2 = gated ? 2 : 1;
    const int per = (NT / 16 + ks - 1) / ks * 16;
    const int st = NT == 128 ? stages_for(128, gated) : NT == 64 ? stages_for(64, gated) : stages_for(32, gated);
    const size_t stage = (size_t)(BM * H2 + 2 * NT) * BK * 2;
    if ((size_t)ks * H2 * BM * (per + 4) * 4 > (size_t)st * stage) return false;
    const int cap = NT == 128 ? (gated ? cluster_capacity<128, true>(ks) : cluster_capacity<128, false>(ks))
                  : NT == 64 ? (gated ? cluster_capacity<64, true>(ks) : cluster_capacity<64, false>(ks))
                             : (gated ? cluster_capacity<32, true>(ks) : cluster_capacity<32, false>(ks));
    return cap > 0;
}
#endif

cudaError_t launch_linear_tc(const void* W, int N, int K, const float* X, int ldx, int M, float* Y, int ldy,
                             const float* bias, int accumulate, const TcScratch& tc, int* err, cudaStream_t st) {
    int nt = 32, ks = 1;
    pick_shape<false>(N, M, K, &nt, &ks);
    switch (nt) {
        case 128: return launch_tc<128, false>(W, N, K, X, ldx, M, Y, ldy, bias, accumulate, 0, nullptr, 0, ks, tc, err, st);
        case 64: return launch_tc<64, false>(W, N, K, X, ldx, M, Y, ldy, bias, accumulate, 0, nullptr, 0, ks, tc, err, st);
        default: return launch_tc<32, false>(W, N, K, X, ldx, M, Y, ldy, bias, accumulate, 0, nullptr, 0, ks, tc, err, st);
    }
}

cudaError_t launch_linear_gated_tc(const void* W, int F, int K, const float* X, int ldx, int M, float* out, int ldo,
                                   const TcScratch& tc, int* err, cudaStream_t st, const TcScratch* out_split) {
    int nt = 32, ks = 1;
    pick_shape<true>(F, M, K, &nt, &ks);
    switch (nt) {
        case 128: return launch_tc<128, true>(W, F, K, X, ldx, M, nullptr, 0, nullptr, 0, F, out, ldo, ks, tc, err, st, out_split);
        case 64: return launch_tc<64, true>(W, F, K, X, ldx, M, nullptr, 0, nullptr, 0, F, out, ldo, ks, tc, err, st, out_split);
        default: return launch_tc<32, true>(W, F, K, X, ldx, M, nullptr, 0, nullptr, 0, F, out, ldo, ks, tc, err, st, out_split);
    }
}

}  // namespace q3
