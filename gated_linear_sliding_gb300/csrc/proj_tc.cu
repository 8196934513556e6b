// The projections in front of the Lizard token mixer on the tensor cores (sm_103a).
//
// Lizard summary (gist.science/ko/paper/2507.09025), sec. 2-A-1: the gate is a learned
// projection of the layer input, Gamma_i = sigmoid(W_gamma x_i), next to the attention
// projections.  One GEMM produces all four inputs of the mixer,
//   [q | k | v | g] = x W^T          x [T, dm], W [N, dm], N = Hq d + 2 Hkv d + Hkv D,
// and two more give its gradients from the mixer's dq, dk, dv, dg (dY = [dq | dk | dv | dg]):
//   dx = dY W,   dW = dY^T x.
//
// One persistent kernel serves the three: C[M, N] = sum_k A[m, k] B[n, k] over 128 x BN tiles,
// with A and B each stored K-major or MN-major in global memory.  Warp 0 (one lane) streams
// A and B tiles by TMA into a ring of shared-memory stages (128-byte swizzle), warp 1 (one
// lane) issues the tcgen05 MMAs into one of two TMEM accumulators, and warps 2..5 drain the
// other accumulator to global memory, so a tile's epilogue overlaps the next tile's MMAs.
// A may come in up to four pieces (the four gradient tensors) split along K or along M, and
// C may go out in up to four pieces split along N (q, k, v, g).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"
#include "tc_util.cuh"

namespace lz {
namespace {

using namespace sm100;
using namespace tc;

constexpr int PBM = 128;   // tile rows (MMA M)
constexpr int PBK = 64;    // K per stage: one 128-byte swizzle atom of bf16
constexpr int PNT = 192;   // 6 warps: copies, MMAs, 4 x epilogue

struct GemmArgs {
    CUtensorMap a[4];       // pieces of A
    CUtensorMap b;
    int64_t M, N, K;
    int64_t a_lo[5];        // piece p covers [a_lo[p], a_lo[p + 1]) along K (a_split_k) or M
    int a_np, a_split_k, a_mn, b_mn;
    void* c[4];             // pieces of C along N, row strides c_ld (elements)
    int64_t c_lo[5], c_ld[4];
    int c_np, out_f32;
    WsHeader* hdr;
};

template <int BN, int NS>
struct PSmem {
    static constexpr uint32_t A = PBM * PBK * 2;  // 16 KB
    static constexpr uint32_t B = BN * PBK * 2;
    static constexpr uint32_t STAGE = A + B;
    static constexpr uint32_t BARS = NS * STAGE;
    static constexpr uint32_t BYTES = BARS + 256 + 1024;
};

__device__ __forceinline__ int piece_of(const int64_t* lo, int np, int64_t x) {
    int p = 0;
    while (p + 1 < np && x >= lo[p + 1]) ++p;
    return p;
}

// Bounded wait; on failure record the timeout once and raise the CTA's abort flag.
__device__ __forceinline__ bool pwait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                      WsHeader* hdr, unsigned where) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort) return false;
        if (clock64() - t0 > kTimeout) {
            if (atomicExch((int*)abort, 1) == 0) report(hdr, LIZARD_ERR_TIMEOUT, where);
            return false;
        }
    }
    return true;
}

template <int BN, int NS>
__global__ void __launch_bounds__(PNT, 1) proj_gemm_kernel(const __grid_constant__ GemmArgs g) {
    using L = PSmem<BN, NS>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::BARS);
    uint64_t* empty = full + NS;
    uint64_t* acc_full = empty + NS;
    uint64_t* acc_empty = acc_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t ntm = (g.M + PBM - 1) / PBM, ntn = (g.N + BN - 1) / BN;
    const int64_t ntiles = ntm * ntn;
    const int nk = (int)((g.K + PBK - 1) / PBK);

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 128);
        }
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 2 * BN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // producer: A and B tiles of every K step of every tile of this CTA
            for (int i = 0; i < 4; ++i)
                if (i < g.a_np) prefetch_tmap(&g.a[i]);
            prefetch_tmap(&g.b);
            uint32_t gk = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const int64_t m0 = (t / ntn) * PBM, n0 = (t % ntn) * BN;
                const int pm = g.a_split_k ? 0 : piece_of(g.a_lo, g.a_np, m0);
                for (int kt = 0; kt < nk; ++kt, ++gk) {
                    const int s = (int)(gk % NS);
                    const uint32_t ph = (gk / NS) & 1u;
                    if (!pwait(&empty[s], ph ^ 1u, abort, g.hdr, 80)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = sm + s * L::STAGE;
                    uint8_t* sb = sa + L::A;
                    const int64_t k0 = (int64_t)kt * PBK;
                    mbar_arrive_expect_tx(&full[s], L::STAGE);
                    const int p = g.a_split_k ? piece_of(g.a_lo, g.a_np, k0) : pm;
                    if (!g.a_mn) {  // A K-major: [rows][K]
                        const int ka = (int)(g.a_split_k ? k0 - g.a_lo[p] : k0);
                        tma_load_2d(sa, &g.a[p], &full[s], ka, (int)m0);
                    } else {        // A MN-major: [K rows][M], two 64-column blocks
                        const int ma = (int)(m0 - g.a_lo[p]);
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            tma_load_2d(sa + h * 8192, &g.a[p], &full[s], ma + 64 * h, (int)k0);
                    }
                    if (!g.b_mn) {
                        tma_load_2d(sb, &g.b, &full[s], (int)k0, (int)n0);
                    } else {
#pragma unroll
                        for (int h = 0; h < BN / 64; ++h)
                            tma_load_2d(sb + h * 8192, &g.b, &full[s], (int)n0 + 64 * h, (int)k0);
                    }
                }
            }
            // on an abort, let the copies already issued land before the CTA exits
            if (!ok) {
                const uint32_t last = gk;
                for (uint32_t q = last > (uint32_t)NS ? last - NS : 0; q < last; ++q)
                    mbar_wait(&full[q % NS], (q / NS) & 1u, kTimeout);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // MMA issue: one accumulator per tile, alternating
            const uint32_t idesc = idesc_bf16(PBM, BN, g.a_mn != 0, g.b_mn != 0);
            uint32_t gk = 0;
            int it = 0;
            bool ok = true, out = false;
            for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++it) {
                const int ab = it & 1;
                if (!pwait(&acc_empty[ab], ((it >> 1) & 1) ^ 1u, abort, g.hdr, 81)) break;
                tc_fence_after();
                const uint32_t acc = tb + (uint32_t)(ab * BN);
                for (int kt = 0; kt < nk; ++kt, ++gk) {
                    const int s = (int)(gk % NS);
                    if (!pwait(&full[s], (gk / NS) & 1u, abort, g.hdr, 82)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = base + s * L::STAGE, sb = sa + L::A;
                    const uint64_t da = g.a_mn ? mndesc(sa, 8192) : kdesc(sa);
                    const uint64_t db = g.b_mn ? mndesc(sb, 8192) : kdesc(sb);
#pragma unroll
                    for (int j = 0; j < PBK / 16; ++j) {
                        // K step of 16: 32 bytes along a K-major row, 16 rows of an MN-major tile
                        const uint64_t oa = g.a_mn ? (uint64_t)((j * 2048) >> 4) : (uint64_t)((j * 32) >> 4);
                        const uint64_t ob = g.b_mn ? (uint64_t)((j * 2048) >> 4) : (uint64_t)((j * 32) >> 4);
                        mma_bf16(acc, da + oa, db + ob, idesc, (kt > 0 || j > 0) ? 1u : 0u);
                    }
                    mma_commit(&empty[s]);  // the stage is free once these MMAs have read it
                    out = true;
                }
                if (!ok) break;
                mma_commit(&acc_full[ab]);
            }
            if (out && !ok) {  // drain what was issued before the abort
                mma_commit(&acc_full[(it & 1)]);
                mbar_wait(&acc_full[it & 1], (it >> 1) & 1u, kTimeout);
            }
        }
        __syncwarp();
    } else {
        // epilogue: TMEM lanes 32 (warp mod 4) .. + 31 are this warp's rows
        const int quad = warp & 3;
        const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
        int it = 0;
        for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
            const int ab = it & 1;
            const bool got = pwait(&acc_full[ab], (it >> 1) & 1u, abort, g.hdr, 83);
            if (!got) break;
            tc_fence_after();
            const int64_t m0 = (t / ntn) * PBM, n0 = (t % ntn) * BN;
            const int64_t m = m0 + 32 * quad + lane;
            const int p = piece_of(g.c_lo, g.c_np, n0);
            const int64_t ncol = n0 - g.c_lo[p];
#pragma unroll 1
            for (int ch = 0; ch < BN / 32; ++ch) {
                float v[32];
                tmem_ld32(tb + lane_off + (uint32_t)(ab * BN + 32 * ch), v);
                tmem_wait_ld();
                const int64_t n = n0 + 32 * ch;
                if (m < g.M && n < g.N) {
                    if (g.out_f32) {
                        float* dst = (float*)g.c[p] + m * g.c_ld[p] + ncol + 32 * ch;
#pragma unroll
                        for (int k = 0; k < 32; k += 4)
                            *reinterpret_cast<float4*>(dst + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
                    } else {
                        __nv_bfloat16* dst = (__nv_bfloat16*)g.c[p] + m * g.c_ld[p] + ncol + 32 * ch;
#pragma unroll
                        for (int k = 0; k < 32; k += 8)
                            *reinterpret_cast<uint4*>(dst + k) =
                                make_uint4(pack_bf16(v[k], v[k + 1]), pack_bf16(v[k + 2], v[k + 3]),
                                           pack_bf16(v[k + 4], v[k + 5]), pack_bf16(v[k + 6], v[k + 7]));
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[ab]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tb, 2 * BN);
    }
}

// 2-D bf16 tensor map of a row-major [rows, cols] array, box {64, box_rows}, 128-byte swizzle.
bool map2d(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t str[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    return make_map(m, ptr, 2, dims, str, box);
}

template <int BN, int NS>
cudaError_t run_gemm(const GemmArgs& g, cudaStream_t s) {
    using L = PSmem<BN, NS>;
    int dev = 0, nsm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(proj_gemm_kernel<BN, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)L::BYTES);
    if (e != cudaSuccess) return e;
    const int64_t tiles = ((g.M + PBM - 1) / PBM) * ((g.N + BN - 1) / BN);
    const unsigned grid = (unsigned)(tiles < nsm ? tiles : nsm);
    if (grid == 0) return cudaSuccess;
    proj_gemm_kernel<BN, NS><<<grid, PNT, L::BYTES, s>>>(g);
    return cudaGetLastError();
}

cudaError_t gemm(const GemmArgs& g, int bn, cudaStream_t s) {
    return bn == 256 ? run_gemm<256, 4>(g, s) : run_gemm<128, 6>(g, s);
}

}  // namespace

bool proj_supported(const Plan& p, int64_t dm, int* bn) {
    if (p.dtype != LIZARD_BF16 || dm < 64 || dm % 64 != 0 || dm > (int64_t)1 << 24) return false;
    const int64_t w[4] = {p.Hq * p.d, p.Hkv * p.d, p.Hkv * p.d, p.Hkv * p.D};
    bool all256 = true;
    for (int i = 0; i < 4; ++i) {
        if (w[i] % 128 != 0) return false;
        all256 = all256 && (w[i] % 256 == 0);
    }
    if (p.B * p.L >= ((int64_t)1 << 31)) return false;
    *bn = all256 ? 256 : 128;
    return encode_fn() != nullptr;
}

cudaError_t launch_proj_fwd(const Plan& p, int64_t dm, const void* x, const void* W, void* q,
                            void* k, void* v, void* gl, void* hdr, cudaStream_t s) {
    int bn = 128;
    if (!proj_supported(p, dm, &bn)) return cudaErrorInvalidValue;
    const int64_t T = p.B * p.L;
    const int64_t w[4] = {p.Hq * p.d, p.Hkv * p.d, p.Hkv * p.d, p.Hkv * p.D};
    GemmArgs g{};
    g.M = T;
    g.N = w[0] + w[1] + w[2] + w[3];
    g.K = dm;
    if (!map2d(&g.a[0], x, T, dm, PBM)) return cudaErrorInvalidValue;
    if (!map2d(&g.b, W, g.N, dm, bn)) return cudaErrorInvalidValue;
    g.a_np = 1;
    g.a_lo[0] = 0;
    g.a_lo[1] = dm;
    g.a_split_k = 1;
    g.a_mn = g.b_mn = 0;
    void* outs[4] = {q, k, v, gl};
    g.c_np = 4;
    g.c_lo[0] = 0;
    for (int i = 0; i < 4; ++i) {
        g.c[i] = outs[i];
        g.c_ld[i] = w[i];
        g.c_lo[i + 1] = g.c_lo[i] + w[i];
    }
    g.out_f32 = 0;
    g.hdr = (WsHeader*)hdr;
    return gemm(g, bn, s);
}

cudaError_t launch_proj_bwd(const Plan& p, int64_t dm, const void* x, const void* W,
                            const void* dq, const void* dk, const void* dv, const void* dg,
                            void* dx, float* dW, void* hdr, cudaStream_t s) {
    int bn = 128;
    if (!proj_supported(p, dm, &bn)) return cudaErrorInvalidValue;
    const int64_t T = p.B * p.L;
    const int64_t w[4] = {p.Hq * p.d, p.Hkv * p.d, p.Hkv * p.d, p.Hkv * p.D};
    const void* dys[4] = {dq, dk, dv, dg};
    const int64_t N = w[0] + w[1] + w[2] + w[3];
    // dx [T, dm] = dY [T, N] W [N, dm]: A = the four dY pieces along K (K-major), B = W MN-major
    {
        GemmArgs g{};
        g.M = T;
        g.N = dm;
        g.K = N;
        g.a_np = 4;
        g.a_split_k = 1;
        g.a_lo[0] = 0;
        for (int i = 0; i < 4; ++i) {
            if (!map2d(&g.a[i], dys[i], T, w[i], PBM)) return cudaErrorInvalidValue;
            g.a_lo[i + 1] = g.a_lo[i] + w[i];
        }
        if (!map2d(&g.b, W, N, dm, 64)) return cudaErrorInvalidValue;
        g.a_mn = 0;
        g.b_mn = 1;
        g.c_np = 1;
        g.c[0] = dx;
        g.c_ld[0] = dm;
        g.c_lo[0] = 0;
        g.c_lo[1] = dm;
        g.out_f32 = 0;
        g.hdr = (WsHeader*)hdr;
        const cudaError_t e = gemm(g, dm % 256 == 0 ? 256 : 128, s);
        if (e != cudaSuccess) return e;
    }
    // dW [N, dm] = dY^T [N, T] x [T, dm]: A = the dY pieces along M (MN-major), B = x MN-major
    {
        GemmArgs g{};
        g.M = N;
        g.N = dm;
        g.K = T;
        g.a_np = 4;
        g.a_split_k = 0;
        g.a_lo[0] = 0;
        for (int i = 0; i < 4; ++i) {
            if (!map2d(&g.a[i], dys[i], T, w[i], 64)) return cudaErrorInvalidValue;
            g.a_lo[i + 1] = g.a_lo[i] + w[i];
        }
        if (!map2d(&g.b, x, T, dm, 64)) return cudaErrorInvalidValue;
        g.a_mn = 1;
        g.b_mn = 1;
        g.c_np = 1;
        g.c[0] = dW;
        g.c_ld[0] = dm;
        g.c_lo[0] = 0;
        g.c_lo[1] = dm;
        g.out_f32 = 1;
        g.hdr = (WsHeader*)hdr;
        return gemm(g, dm % 256 == 0 ? 256 : 128, s);
    }
}

}  // namespace lz
