// Device-side shared definitions for the q3tts kernels (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "q3tts.h"

namespace q3 {

using bf16 = __nv_bfloat16;

constexpr int HD = 128;              // head_dim (fixed by the method)
constexpr int MAX_GROUPS = 16;       // codebooks per frame
constexpr int MAX_VOCAB = 4096;      // largest codec / predictor vocabulary
constexpr int SEEN_WORDS = MAX_VOCAB / 32;

// Device error word bits (OR-ed in; read once per call on the host).
constexpr int ERRB_NAN = 1;
constexpr int ERRB_BOUNDS = 2;
constexpr int ERRB_TIMEOUT = 4;
constexpr int ERRB_LAUNCH = 8;   // a kernel found itself launched in a shape it cannot serve

// Per-row decode state, resident in the workspace.
struct RowState {
    int pos;        // next talker position
    int sel;        // talker selections made; the next one is selection `sel`
    int code0;      // last codebook-0 selection (pending: its frame is not complete yet)
    int finished;
    int reason;     // Q3_RUNNING / Q3_FINISHED_*
    int frames;     // frames completed
    int n_text;     // trailing text rows
    int text_off;   // first text row in the workspace text buffer
    int pad_[8];
    uint32_t seen[SEEN_WORDS];  // codebook-0 ids selected so far (repetition penalty)
};

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(bf16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// 16-byte streaming load that does not allocate in L1 (weights are read once).
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float (&v)[8]) {
    v[0] = __uint_as_float(u.x << 16); v[1] = __uint_as_float(u.x & 0xffff0000u);
    v[2] = __uint_as_float(u.y << 16); v[3] = __uint_as_float(u.y & 0xffff0000u);
    v[4] = __uint_as_float(u.z << 16); v[5] = __uint_as_float(u.z & 0xffff0000u);
    v[6] = __uint_as_float(u.w << 16); v[7] = __uint_as_float(u.w & 0xffff0000u);
}

// 8 consecutive elements (index multiple of 8) as fp32, weight stream.
__device__ __forceinline__ void load8_stream(const bf16* p, float (&v)[8]) { unpack_bf16x8(ld_stream_u4(p), v); }
__device__ __forceinline__ void load8_stream(const float* p, float (&v)[8]) {
    uint4 a = ld_stream_u4(p), b = ld_stream_u4(p + 4);
    v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y); v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
    v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y); v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
}
// 8 consecutive elements, cached (activations, KV).
__device__ __forceinline__ void load8(const bf16* p, float (&v)[8]) { unpack_bf16x8(*(const uint4*)p, v); }
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
    float4 a = *(const float4*)p, b = *((const float4*)p + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

}  // namespace q3
