// Self-test of the bounded-wait failure path used by the tensor-core kernels.
//
// One CTA allocates TMEM, waits on an mbarrier that nothing ever arrives at, gives up
// after `limit_cycles` SM cycles exactly as the forward kernel's waits do, records
// LIZARD_ERR_TIMEOUT in the workspace status word, frees its TMEM and returns.  The
// GPU context stays usable; the host reads the status with lizard_read_device_status.
#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace lz {
namespace {

using namespace sm100;

__global__ void __launch_bounds__(32) wait_timeout_probe(WsHeader* hdr, long long limit_cycles) {
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    tmem_alloc(&tmem, 32);
    tmem_relinquish();
    __syncwarp();
    tc_fence_after();
    // phase 0 never completes: no thread arrives and no copy is in flight
    const bool ok = mbar_wait(&bar, 0, limit_cycles);
    if (!ok && threadIdx.x == 0) report(hdr, LIZARD_ERR_TIMEOUT, 0xFFu);
    tc_fence_before();
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 32);
}

}  // namespace
}  // namespace lz

using namespace lz;

extern "C" lizard_status lizard_selftest_wait_timeout(void* workspace, size_t ws_bytes,
                                                       long long limit_cycles, void* stream) {
    if (limit_cycles < 0 || limit_cycles > 4000000000LL) return LIZARD_ERR_INVALID_ARG;
    if (workspace == nullptr) {
        // the status word of lizard_attn_fwd_noalloc's fixed scratch (current device)
        if (noalloc_header(&workspace) != cudaSuccess) return LIZARD_ERR_CUDA;
        ws_bytes = kHeaderBytes;
    }
    if (((uintptr_t)workspace & 15u) != 0) return LIZARD_ERR_INVALID_ARG;
    if (ws_bytes < kHeaderBytes) return LIZARD_ERR_WORKSPACE;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return LIZARD_ERR_CUDA;
    if (!(major == 10 && minor == 3)) return LIZARD_ERR_UNSUPPORTED;
    wait_timeout_probe<<<1, 32, 0, (cudaStream_t)stream>>>((WsHeader*)workspace, limit_cycles);
    return cudaGetLastError() == cudaSuccess ? LIZARD_OK : LIZARD_ERR_CUDA;
}
