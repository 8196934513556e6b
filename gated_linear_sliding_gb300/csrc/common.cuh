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
