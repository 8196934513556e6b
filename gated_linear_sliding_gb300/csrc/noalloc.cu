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

bool aligned16_na(const void* ptr) { return ((uintptr_t)ptr & 15u) == 0; }

}  // namespace
}  // namespace lz

using namespace lz;

extern "C" lizard_status lizard_attn_fwd_noalloc(const lizard_dims* dims, const void* q,
                                                 const void* k, const void* v, const void* g,
                                                 const void* Wf, const float* sinks, void* y,
                                                 float* lse, float* S_out, float* z_out,
                                                 void* kcache_out, void* vcache_out,
                                                 void* stream) {
    Plan p;
    if (!make_plan(dims, &p)) return LIZARD_ERR_INVALID_ARG;
    // scratch this problem needs (checked first: it depends on the dimensions only): the
    // status word, plus one boundary-state record per (segment, batch x KV head) when the
    // sequence is split into several segments, counted with the segmentation the launch
    // below will use
    Plan pl = p;
    if (fwd_tc_supported(p)) fwd_tc_plan(&pl);
    const size_t need =
        kHeaderBytes +
        (pl.P > 1 ? sizeof(float) * (size_t)(pl.rec_step * (pl.P - 1) + 1) *
                        (size_t)(p.B * p.Hkv) * p.rec_floats
                  : 0);
    if (need > kNoAllocScratchBytes) return LIZARD_ERR_WORKSPACE;
    if (!q || !k || !v || !g || !Wf || !y || (p.M > 0 && !sinks)) return LIZARD_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, g, Wf, sinks, y, lse, S_out, z_out, kcache_out, vcache_out};
    for (const void* ptr : ptrs)
        if (ptr && !aligned16_na(ptr)) return LIZARD_ERR_INVALID_ARG;
    if ((S_out == nullptr) != (z_out == nullptr)) return LIZARD_ERR_INVALID_ARG;
    if ((kcache_out == nullptr) != (vcache_out == nullptr)) return LIZARD_ERR_INVALID_ARG;
    if (!((p.d == 64 || p.d == 128) && (p.D == 64 || p.D == 128) && p.B * p.Hkv <= 65535 &&
          p.B * p.Hq <= ((int64_t)1 << 30)))
        return LIZARD_ERR_UNSUPPORTED;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LIZARD_ERR_CUDA;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return LIZARD_ERR_CUDA;
    if (!(major == 10 && minor == 3)) return LIZARD_ERR_UNSUPPORTED;

    void* scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess) return LIZARD_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    // the array keeps the previous call's contents: the status word must start at zero
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
    cudaError_t e = fwd_tc_supported(p) ? launch_fwd_tc(p, a, s) : launch_fwd_simt(p, a, s);
    if (e == cudaSuccess && kcache_out != nullptr)
        e = launch_ring_fill(p, k, v, kcache_out, vcache_out, s);
    return e == cudaSuccess ? LIZARD_OK : LIZARD_ERR_CUDA;
}
