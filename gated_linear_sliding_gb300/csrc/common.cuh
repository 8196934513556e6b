// Device helpers shared by the Lizard kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lizard.h"

namespace lz {

// Element access for the two storage types.
__device__ __forceinline__ float ld(const float* p) { return *p; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st(float* p, float x) { *p = x; }
__device__ __forceinline__ void st(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// Exponential: the fp32 path keeps CUDA's accurate expf; the bf16 path uses the
// fast hardware approximation, whose error is far below bf16 resolution.
template <bool FAST>
__device__ __forceinline__ float ex(float x) {
    if constexpr (FAST) return __expf(x);
    else return expf(x);
}

// log(sigmoid(x)) = -softplus(-x), evaluated without overflow for any x.
template <bool FAST>
__device__ __forceinline__ float log_sigmoid(float x) {
    float a = fminf(x, 0.0f);
    return a - log1pf(ex<FAST>(-fabsf(x)));
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// Lower clamp of the per-row exponent shift of the shared normaliser: keeps the
// state terms' factor e^{-m} below e^{60}.
constexpr float kMinShift = -60.0f;

// Programmatic dependent launch.  A kernel launched with launch_dependent() may start while
// the previous kernel of the stream still runs: it must call grid_dep_wait() before it reads
// anything that kernel writes (a no-op when the launch carried no such dependency).  A kernel
// calls grid_dep_launch() to let the next one be launched before it completes.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Device status word at the head of every workspace.
struct WsHeader {
    unsigned int status;
    unsigned int where;
    unsigned int pad[62];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

__device__ __forceinline__ void report(WsHeader* h, unsigned int code, unsigned int where) {
    if (h != nullptr && atomicCAS(&h->status, 0u, code) == 0u) h->where = where;
}

}  // namespace lz
