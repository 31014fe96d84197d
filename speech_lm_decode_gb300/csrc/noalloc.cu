// q3tts_sample_logits_noalloc: the logits processors and draw on caller-given
// logits without a handle and without any device allocation.
//
// Who needs it: code that cannot call cudaMalloc (or have a framework allocate
// for it) at the point where it wants a draw -- for example a caller running
// inside another library's allocator callback, a real-time audio thread that
// must not block on the allocator, or a process whose device memory is fully
// reserved by another runtime.  Such callers still own their inputs and
// outputs; the only device memory this entry point needs besides them is a
// small staging area, which lives in the fixed array below.
//
// The staging area is one file-scope __device__ array per GPU that loads this
// library.  It is created when the module is loaded and kept until the process
// exits (QN_MAX_SETS sets at most per call, about 70 KB).  Host code cannot use
// the array's name as a device address, so the first call on each device looks
// the address up with cudaGetSymbolAddress (with that device current) and
// caches it.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace q3 {
namespace {

constexpr int QN_MAX_SETS = 1024;

// Layout of the staging area (every call overwrites it).
struct NoAllocScratch {
    q3tts_sampling params[QN_MAX_SETS];
    int32_t sel[QN_MAX_SETS];
    int32_t row[QN_MAX_SETS];
    int32_t ids[QN_MAX_SETS];
    int err;
};

static __device__ __align__(256) unsigned char g_noalloc_scratch[sizeof(NoAllocScratch)];

constexpr int MAX_DEVICES = 64;
std::mutex g_lock;
NoAllocScratch* g_dev_ptr[MAX_DEVICES] = {};

// Device address of the staging area on the current device (looked up once).
cudaError_t scratch_for_current_device(NoAllocScratch** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(g_lock);
    if (!g_dev_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_dev_ptr[dev] = static_cast<NoAllocScratch*>(p);
    }
    *out = g_dev_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace q3

using namespace q3;

extern "C" int q3tts_sample_logits_noalloc(int n, int vocab, const float* logits, int talker,
                                           const q3tts_sampling* params, const uint8_t* seen,
                                           const int32_t* sel_index, int step, const int32_t* noise_row, int eos_id,
                                           int suppress_lo, int suppress_hi, int32_t* ids_out, void* stream) {
    if (n < 0 || n > QN_MAX_SETS) return Q3_ERR_CAPACITY;
    if (n == 0) return Q3_OK;
    if (vocab < 2 || vocab > MAX_VOCAB || !logits || !params || !sel_index || !noise_row || !ids_out)
        return Q3_ERR_ARG;
    if (talker && (eos_id < 0 || eos_id >= vocab || suppress_lo < 0 || suppress_hi > vocab || suppress_lo > suppress_hi))
        return Q3_ERR_ARG;
    for (int i = 0; i < n; ++i)
        if (!sampling_ok(params[i], talker != 0)) return Q3_ERR_ARG;
    NoAllocScratch* s = nullptr;
    if (scratch_for_current_device(&s) != cudaSuccess) return Q3_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    if (sampler_init() != cudaSuccess) return Q3_ERR_CUDA;
    // the previous call's contents stay in the area: the error word must start at zero
    if (cudaMemsetAsync(&s->err, 0, sizeof(int), st) != cudaSuccess) return Q3_ERR_CUDA;
    if (cudaMemcpyAsync(s->params, params, (size_t)n * sizeof(q3tts_sampling), cudaMemcpyHostToDevice, st) !=
            cudaSuccess ||
        cudaMemcpyAsync(s->sel, sel_index, (size_t)n * sizeof(int32_t), cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(s->row, noise_row, (size_t)n * sizeof(int32_t), cudaMemcpyHostToDevice, st) != cudaSuccess)
        return Q3_ERR_CUDA;
    if (launch_sample_sets(logits, n, vocab, talker, s->params, seen, s->sel, step, s->row, eos_id, suppress_lo,
                           suppress_hi, s->ids, &s->err, st) != cudaSuccess)
        return Q3_ERR_CUDA;
    int err = 0;
    if (cudaMemcpyAsync(ids_out, s->ids, (size_t)n * sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemcpyAsync(&err, &s->err, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return Q3_ERR_CUDA;
    return (err & ERRB_NAN) ? Q3_ERR_NAN : Q3_OK;
}
