// Allocation-free base projection for decode-sized batches.
//
// Some callers cannot allocate device memory at the moment they need a
// projection: code that runs inside a CUDA stream capture (cudaMalloc and
// cudaFree cannot be captured and break the capture), plugins hosted by another
// runtime that owns the whole device-memory budget and forbids allocations after
// start-up, and latency-critical loops that cannot afford the device-wide
// synchronisation an allocation may cause.  Such callers cannot create an adapter
// pool, whose workspace comes from cudaMalloc.  This entry point runs the split-K
// tensor-core projection of the decode path with its scratch -- the fp32 partial
// tiles of the K splits, their arrival counters and a status word -- in one
// file-scope device array instead.  Every GPU that loads the library holds that
// array (NOALLOC_SCRATCH_BYTES, about 8 MiB) until the process exits.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>

#include "../../include/mlora.h"
#include "internal.h"
#include "tc.h"

namespace mlora {

constexpr size_t NOALLOC_PARTIAL_BYTES = 8u << 20;   // fp32 partial tiles of the K splits
constexpr int NOALLOC_MAX_TILES = 2048;              // one counter per 128 output features: dout <= 262144
constexpr size_t NOALLOC_SCRATCH_BYTES = NOALLOC_PARTIAL_BYTES + NOALLOC_MAX_TILES * sizeof(int32_t) + 256;

// Layout: [partials | counters | status word]
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[64];          // device address of g_noalloc_scratch, per device (nullptr = not set up)

mlora_status noalloc_fail(mlora_status s, const std::string& msg) {
    set_last_error(msg);
    return s;
}

// Once per device, with that device current: the kernels' shared-memory caps and
// the device address of the scratch array (its host-side name is not a device address).
mlora_status noalloc_setup(int dev, void** out) {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev]) {
        *out = g_noalloc_ptr[dev];
        return MLORA_OK;
    }
    cudaError_t e = tc_init();
    if (e != cudaSuccess) return noalloc_fail(MLORA_ERR_CUDA, std::string("tc_init: ") + cudaGetErrorString(e));
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr)
        return noalloc_fail(MLORA_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
    g_noalloc_ptr[dev] = ptr;
    *out = ptr;
    return MLORA_OK;
}

}  // namespace
}  // namespace mlora

using namespace mlora;

extern "C" mlora_status mlora_project_noalloc(const void* X, const void* W, int T, int din, int dout, void* Y,
                                              mlora_stream_t stream) {
    if (T == 0) return MLORA_OK;
    if (!X || !W || !Y) return noalloc_fail(MLORA_ERR_INVALID_ARG, "X/W/Y is NULL");
    if (((uintptr_t)X | (uintptr_t)W | (uintptr_t)Y) & 15u)
        return noalloc_fail(MLORA_ERR_INVALID_ARG, "X/W/Y must be 16-byte aligned");
    if (T < 0 || T > 256) return noalloc_fail(MLORA_ERR_UNSUPPORTED, "T must be in [0, 256]");
    if (din < 1 || dout < 1 || din % 8 != 0)
        return noalloc_fail(MLORA_ERR_UNSUPPORTED, "din must be a positive multiple of 8 and dout positive");
    if ((dout + 127) / 128 > NOALLOC_MAX_TILES)
        return noalloc_fail(MLORA_ERR_UNSUPPORTED, "dout exceeds the scratch limit of 262144 output features");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return noalloc_fail(MLORA_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return noalloc_fail(MLORA_ERR_UNSUPPORTED, "device index above 63");
    void* base = nullptr;
    mlora_status st = noalloc_setup(dev, &base);
    if (st != MLORA_OK) return st;
    float* partials = (float*)base;
    int32_t* counters = (int32_t*)((char*)base + NOALLOC_PARTIAL_BYTES);
    uint32_t* status = (uint32_t*)(counters + NOALLOC_MAX_TILES);
    cudaStream_t s = (cudaStream_t)stream;
    // the counters and the status word must start at zero; the array keeps what the last call left
    e = cudaMemsetAsync(counters, 0, NOALLOC_MAX_TILES * sizeof(int32_t) + sizeof(uint32_t), s);
    if (e == cudaSuccess)
        e = tc_project_with_scratch(X, W, T, din, dout, Y, partials, NOALLOC_PARTIAL_BYTES, counters,
                                    NOALLOC_MAX_TILES, status, s);
    if (e != cudaSuccess) return noalloc_fail(MLORA_ERR_CUDA, std::string("launch: ") + cudaGetErrorString(e));
    return MLORA_OK;
}
