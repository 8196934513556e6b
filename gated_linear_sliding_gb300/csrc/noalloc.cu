// lizard_attn_fwd_noalloc: the forward for callers that cannot allocate device memory.
//
// Some callers only ever receive pointers to inputs and outputs: a plugin invoked by
// a host framework that owns every device allocation, or a latency-critical loop that
// must not call cudaMalloc/cudaFree because those may synchronise the whole device.
// This entry point needs no workspace from them.  Its scratch (the status word and
// the per-segment boundary states) lives in one file-scope device array of fixed
// size, which every GPU that loads the library keeps until the process exits.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace lz {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)32 << 20;  // 32 MiB

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[256];  // device address of the array, per device ordinal

// Device address of the scratch array on the current device (looked up once per device,
// with that device current).  Host code must not hand the symbol itself to a kernel.
cudaError_t noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 256) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

// Scratch bytes a call needs: the status word, then the boundary-state records its launch
// uses (the same count as in a caller's workspace), then the reading's scratch (MASKED and
// LAGGED) from the next 256-byte boundary.
size_t noalloc_records_end(const Plan& p, bool tc) {
    return kHeaderBytes +
           sizeof(float) * fwd_records_used(p, tc) * (size_t)(p.B * p.Hkv) * p.rec_floats;
}
size_t noalloc_reading_offset(const Plan& p, bool tc) {
    return (noalloc_records_end(p, tc) + 255) & ~(size_t)255;
}
size_t noalloc_need(const Plan& p, bool tc) {
    const size_t r = reading_scratch_bytes(p);
    return r == 0 ? noalloc_records_end(p, tc) : noalloc_reading_offset(p, tc) + r;
}

}  // namespace

// The status header (first 256 bytes) of the array, for the failure-path self-test.
cudaError_t noalloc_header(void** out) { return noalloc_scratch(out); }

}  // namespace lz

using namespace lz;

extern "C" size_t lizard_attn_fwd_noalloc_scratch(const lizard_dims* dims) {
    Plan p;
    if (!make_plan(dims, &p)) return 0;
    // the larger of the two walks' needs (a masked call returning the state takes the SIMT walk)
    const size_t tc = noalloc_need(p, fwd_uses_tc(p, false));
    const size_t st = noalloc_need(p, fwd_uses_tc(p, true));
    return tc > st ? tc : st;
}

extern "C" lizard_status lizard_attn_fwd_noalloc(const lizard_dims* dims, const void* q,
                                                 const void* k, const void* v, const void* g,
                                                 const void* Wf, const float* sinks, void* y,
                                                 float* lse, float* S_out, float* z_out,
                                                 void* kcache_out, void* vcache_out,
                                                 void* stream) {
    Plan p;
    lizard_status st = fwd_check(dims, &p, q, k, v, g, Wf, sinks, y, lse, S_out, z_out,
                                 kcache_out, vcache_out);
    if (st != LIZARD_OK) return st;
    const bool tc = fwd_uses_tc(p, S_out != nullptr || z_out != nullptr);
    if (noalloc_need(p, tc) > kNoAllocScratchBytes) return LIZARD_ERR_WORKSPACE;
    st = device_status();
    if (st != LIZARD_OK) return st;

    void* scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess) return LIZARD_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    // the array keeps the previous call's contents: the status word must start at zero
    // (boundary records and hand-off marks are always written before they are read)
    if (cudaMemsetAsync(scratch, 0, kHeaderBytes, s) != cudaSuccess) return LIZARD_ERR_CUDA;

    FwdArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.Wf = Wf;
    a.sinks = sinks;
    a.y = y;
    a.lse = lse;
    a.S_out = S_out;
    a.z_out = z_out;
    a.kcache_out = kcache_out;
    a.vcache_out = vcache_out;
    a.header = scratch;
    a.seg = (float*)((char*)scratch + kHeaderBytes);
    a.ev_before = nullptr;
    a.ev_after = nullptr;
    a.rscratch =
        reading_scratch_bytes(p) != 0 ? (char*)scratch + noalloc_reading_offset(p, tc) : nullptr;
    return fwd_launch(p, a, s) == cudaSuccess ? LIZARD_OK : LIZARD_ERR_CUDA;
}

extern "C" lizard_status lizard_read_noalloc_status(void* stream) {
    void* scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess) return LIZARD_ERR_CUDA;
    return lizard_read_device_status(scratch, stream);
}
