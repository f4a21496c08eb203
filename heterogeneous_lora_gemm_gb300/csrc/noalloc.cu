// Allocation-free base projection for decode-sized batches.
//
// Some callers cannot allocate device memory at the moment they need a
// projection: plugins hosted by another runtime that owns the whole device-memory
// budget and forbids allocations after start-up, and latency-critical loops that
// cannot afford the device-wide synchronisation an allocation may cause.  Such callers cannot create an adapter
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
#include "tc_ptx.cuh"

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
    // the counters must start at zero (the array keeps what the last call left); the
    // status word keeps its bits until mlora_project_noalloc_status reads and clears it
    e = cudaMemsetAsync(counters, 0, NOALLOC_MAX_TILES * sizeof(int32_t), s);
    if (e == cudaSuccess)
        e = tc_project_with_scratch(X, W, T, din, dout, Y, partials, NOALLOC_PARTIAL_BYTES, counters,
                                    NOALLOC_MAX_TILES, status, s);
    if (e != cudaSuccess) return noalloc_fail(MLORA_ERR_CUDA, std::string("launch: ") + cudaGetErrorString(e));
    return MLORA_OK;
}

// Status of the allocation-free calls on the current device: synchronizes `stream`,
// reads the status word of the scratch array and clears it.
extern "C" mlora_status mlora_project_noalloc_status(mlora_stream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return noalloc_fail(MLORA_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return noalloc_fail(MLORA_ERR_UNSUPPORTED, "device index above 63");
    void* base = nullptr;
    mlora_status st = noalloc_setup(dev, &base);
    if (st != MLORA_OK) return st;
    uint32_t* status = (uint32_t*)((char*)base + NOALLOC_PARTIAL_BYTES + NOALLOC_MAX_TILES * sizeof(int32_t));
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t word = 0;
    e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&word, status, sizeof word, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, sizeof word, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return noalloc_fail(MLORA_ERR_CUDA, std::string("status read: ") + cudaGetErrorString(e));
    if (word & STATUS_TIMEOUT) return noalloc_fail(MLORA_ERR_DEVICE_TIMEOUT, "a kernel pipeline wait gave up");
    return MLORA_OK;
}

namespace mlora {
namespace {

// One pipeline wait that nothing completes: an mbarrier expecting one arrival that
// never comes, waited on with the kernels' bounded wait and the given limit.  Its
// expiry raises STATUS_TIMEOUT in `status`, as a real pipeline wait that gave up would.
__global__ void noalloc_expire_wait_kernel(uint32_t* status, long long limit) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    ptx::mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    ptx::mbar_wait_limit(&bar, 0, &abort_flag, status, limit);
}

}  // namespace
}  // namespace mlora

extern "C" mlora_status mlora_debug_noalloc_expire_wait(long long cycles, mlora_stream_t stream) {
    if (cycles < 1 || cycles > (1ll << 31)) return noalloc_fail(MLORA_ERR_INVALID_ARG, "cycles not in [1, 2^31]");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return noalloc_fail(MLORA_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return noalloc_fail(MLORA_ERR_UNSUPPORTED, "device index above 63");
    void* base = nullptr;
    mlora_status st = noalloc_setup(dev, &base);
    if (st != MLORA_OK) return st;
    uint32_t* status = (uint32_t*)((char*)base + NOALLOC_PARTIAL_BYTES + NOALLOC_MAX_TILES * sizeof(int32_t));
    noalloc_expire_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(status, cycles);
    e = cudaGetLastError();
    if (e != cudaSuccess) return noalloc_fail(MLORA_ERR_CUDA, std::string("launch: ") + cudaGetErrorString(e));
    return MLORA_OK;
}
