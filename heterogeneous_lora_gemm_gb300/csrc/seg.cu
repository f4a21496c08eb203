// Standalone segment-builder kernel (one CTA of 1024 threads), used by
// mlora_debug_segments, by the fp32 forward and by a bf16 forward with no adapter
// loaded.  The bf16 forward otherwise runs the same builder (seg.cuh) in a CTA of
// its tensor-core shrink's grid.
#include "internal.h"
#include "seg.cuh"

namespace mlora {

namespace {

constexpr int SEG_THREADS = 1024;

__global__ void __launch_bounds__(SEG_THREADS, 1)
seg_build_kernel(const int32_t* __restrict__ row_adapter, int T, const SlotRec* __restrict__ slots, Workspace ws,
                 int S, int P, int max_chunks, int stage_rows) {
    extern __shared__ __align__(16) int smem[];
    const seg::Scratch sc = seg::carve(smem, S, P, stage_rows != 0);
    seg::stage(slots, S, ws, row_adapter, T, max_chunks, sc);
    seg::build(S, P, sc);
}

}  // namespace

SegPlan seg_plan(int S, int warps, int scratch_ints_avail, int T) {
    // as many row ranges as fit the scratch (per-(warp, slot) counters), at most one
    // per warp, with the row map staged if it fits too
    for (int stage = 1; stage >= 0; --stage) {
        const int Ts = stage ? T : 0;
        int P = warps;
        while (P > 1 && seg::scratch_ints(S, P, Ts) > scratch_ints_avail) --P;
        if (seg::scratch_ints(S, P, Ts) <= scratch_ints_avail) return SegPlan{P, stage != 0, seg::scratch_ints(S, P, Ts)};
    }
    return SegPlan{0, false, 0};
}

cudaError_t seg_init() {
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa;
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, seg_build_kernel);
    // static shared memory counts against the same per-block limit
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(seg_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - (int)fa.sharedSizeBytes);
    return e;
}

cudaError_t launch_seg_build(const int32_t* row_adapter, int T, const SlotRec* slots, const Workspace& ws,
                             const PoolDims& d, cudaStream_t st) {
    const SegPlan sp = seg_plan(d.S, SEG_THREADS / 32, (200 * 1024) / 4, T);
    if (sp.P < 1) return cudaErrorInvalidConfiguration;
    const size_t smem = sizeof(int) * (size_t)sp.ints;
    seg_build_kernel<<<1, SEG_THREADS, smem, st>>>(row_adapter, T, slots, ws, d.S, sp.P, d.max_chunks,
                                                   sp.stage_rows ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace mlora
