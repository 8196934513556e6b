// Helpers shared by the tcgen05 kernels (forward and backward): constants, the special-
// function exponential, bf16 rounding of pairs, shared-memory descriptors of 128-byte
// swizzled tiles and the host-side tensor-map encoder.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "sm100.cuh"

namespace lz {
namespace tc {

constexpr long long kTimeout = 2000000000LL;  // SM cycles of a bounded wait (about one second)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// 2^x on the special-function unit (inputs here are finite or -inf, which gives +0)
__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 1/x on the special-function unit (1/inf gives +0)
__device__ __forceinline__ float rcpf(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Round a pair to bf16 (nearest even) in place and return it packed (lo in the low half).
__device__ __forceinline__ uint32_t round_pair(float& lo, float& hi) {
    const uint32_t w = sm100::pack_bf16(lo, hi);
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xFFFF0000u);
    return w;
}

// Split a pair into bf16 high parts and the bf16 rounding of the remainders (packed, lo
// element in the low half): hi + lo carries about 16 bits of mantissa.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    float h0 = x0, h1 = x1;
    hi = round_pair(h0, h1);
    lo = sm100::pack_bf16(x0 - h0, x1 - h1);
}

__device__ __forceinline__ void unpack8(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                                        float* o) {
    const uint32_t w[4] = {w0, w1, w2, w3};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        o[2 * k] = __uint_as_float(w[k] << 16);
        o[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
}

// K-major (or MN-major, with the byte distance between 64-element halves as `lbo`)
// descriptors of 128-byte-swizzled tiles; 8-row groups are 1024 bytes apart.
__device__ __forceinline__ uint64_t kdesc(uint32_t addr) {
    return sm100::make_sdesc(addr, 16, 1024, sm100::kSwizzle128);
}
__device__ __forceinline__ uint64_t mndesc(uint32_t addr, uint32_t lbo) {
    return sm100::make_sdesc(addr, lbo, 1024, sm100::kSwizzle128);
}

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
    }
    return fn;
}

// bf16 tensor map; 128-byte swizzle unless `swizzle` is false.
inline bool make_map(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims,
                     const cuuint64_t* strides, const cuuint32_t* box, bool swizzle = true) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(ptr), dims,
              strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A [128][128] fp32 state record passes between global and shared memory through 64 KB of
// shared memory with coalesced 16-byte accesses; each 512-byte row's 16-byte chunks are
// XOR-swizzled by the row, so the per-thread row accesses (TMEM lane = row, 32 columns per
// thread) are free of bank conflicts.
__device__ __forceinline__ uint32_t rec_off(int r, int c) {
    return (uint32_t)(r * 512 + ((c & ~7) | ((c ^ r) & 7)) * 16);
}
__device__ __forceinline__ void stage_record_in(uint8_t* dst, const float* rec) {
    for (int e = threadIdx.x; e < 128 * 128 / 4; e += blockDim.x)
        *reinterpret_cast<float4*>(dst + rec_off(e >> 5, e & 31)) =
            reinterpret_cast<const float4*>(rec)[e];
}
__device__ __forceinline__ void stage_record_out(float* rec, const uint8_t* src) {
    for (int e = threadIdx.x; e < 128 * 128 / 4; e += blockDim.x)
        reinterpret_cast<float4*>(rec)[e] =
            *reinterpret_cast<const float4*>(src + rec_off(e >> 5, e & 31));
}
// Columns [32 part, 32 part + 32) of staged row `row` (zeros when `have` is false) ...
__device__ __forceinline__ void staged_row_read(const uint8_t* src, bool have, int row, int part,
                                                float (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float4 x = have ? *reinterpret_cast<const float4*>(src + rec_off(row, 8 * part + j))
                              : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        v[4 * j] = x.x;
        v[4 * j + 1] = x.y;
        v[4 * j + 2] = x.z;
        v[4 * j + 3] = x.w;
    }
}
// ... and the same columns written.
__device__ __forceinline__ void staged_row_write(uint8_t* dst, int row, int part,
                                                 const float (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
        *reinterpret_cast<float4*>(dst + rec_off(row, 8 * part + j)) =
            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
}

}  // namespace tc
}  // namespace lz
