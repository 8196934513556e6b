// Tensor-core backward of the sliding-window part of the Lizard token mixer on sm_103a
// (tcgen05 MMAs with TMEM accumulators, TMA operands in 128-byte-swizzled shared memory).
//
// Lizard summary (gist.science/ko/paper/2507.09025), sec. 2-A-2: inside the window the
// weights are softmax terms e^{s q_i.k_j} that share the row's normaliser.  With
// lse_i = log of the row's full denominator (times e^{m_i}) and delta_i = dy_i . y_i:
//   p_ij  = e^{s q_i.k_j - lse_i},   j in (i - w, i],
//   ds_ij = s p_ij (dy_i . v_j - delta_i),
//   dq_i += sum_j ds_ij k_j,   dk_j += sum_i ds_ij q_i,   dv_j += sum_i p_ij dy_i.
// The state parts of dq, dk, dv are written first by the SIMT walks; these kernels add the
// window parts on top.
//
// Rows of a query tile are (token, head) pairs of one KV-head group, row = 4 token + head
// (32 tokens x 4 heads = 128 MMA rows), exactly the order a TMA box {d, 4 heads, 32 tokens}
// lands in shared memory.
//   bwd_win_kv_tc: one CTA per (128-key tile, batch x KV head); the keys are the MMA rows:
//     S^T = K Q^T and dP^T = V dY^T per query tile, then P^T and dS^T (bf16, in TMEM) feed
//     dV += P^T dY and dK += dS^T Q.
//   bwd_win_q_tc: one CTA per (128-token query block, batch x KV head); the query rows are
//     the MMA rows: S = Q K^T, dP = dY V^T against the 128 keys that can reach the tile, then
//     dQ = dS K.
#include <cuda.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"
#include "tc_util.cuh"

namespace lz {
namespace {

using namespace sm100;
using namespace tc;

constexpr int NT = 512;   // 16 warps: warp w owns TMEM lanes 32(w%4).., w/4 picks a 32-column part
constexpr int CT = 32;    // tokens per query tile
constexpr int GQ = 4;     // query heads per KV head
constexpr int DH = 128;   // head dim
constexpr int WIN = 64;   // window
constexpr uint32_t kTile = 32768;  // one 128-row x 128-d bf16 tile (two 64-column halves)

struct Bars {
    uint64_t bar_kv, bar_in[2], bar_s, bar_o, bar_fin;
    uint32_t tmem;
    volatile int abort;
};

// Bounded wait by every thread; all return the same answer.
__device__ __forceinline__ bool all_wait(uint64_t* bar, uint32_t ph, Bars& S, WsHeader* hdr,
                                         unsigned where) {
    bool fail = false;
    if (!mbar_try_wait(bar, ph)) {
        const long long t0 = clock64();
        while (!mbar_try_wait(bar, ph)) {
            if (S.abort || clock64() - t0 > kTimeout) {
                fail = true;
                break;
            }
        }
    }
    if (fail && !S.abort) {
        S.abort = 1;
        report(hdr, LIZARD_ERR_TIMEOUT, where);
    }
    return !__syncthreads_or(fail);
}

__device__ __forceinline__ void quad_sync(int quad) {
    asm volatile("bar.sync %0, 128;" ::"r"(1 + quad) : "memory");
}

// Query and dy tiles of one 32-token chunk (rows 4 token + head) on one barrier phase.
__device__ __forceinline__ void load_qdy(uint8_t* q, uint8_t* dy, const CUtensorMap* tmQ,
                                         const CUtensorMap* tmD, uint64_t* bar, int64_t kv,
                                         int64_t c, int64_t b) {
    mbar_arrive_expect_tx(bar, 2 * kTile);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
        tma_load_4d(q + kb * 16384, tmQ, bar, 64 * kb, (int)(kv * GQ), (int)(c * CT), (int)b);
        tma_load_4d(dy + kb * 16384, tmD, bar, 64 * kb, (int)(kv * GQ), (int)(c * CT), (int)b);
    }
}

// Wait for whatever this thread issued before leaving after an abort.
__device__ __forceinline__ void drain(Bars& S, bool mma_out, uint64_t* tbar, uint32_t tph) {
    mbar_wait(&S.bar_kv, 0, kTimeout);
    if (mma_out) {
        mma_commit(&S.bar_fin);
        mbar_wait(&S.bar_fin, 0, kTimeout);
    }
    if (tbar != nullptr) mbar_wait(tbar, tph, kTimeout);
}

// Add a 32-column fp32 slice to a bf16 row (the state part already there, or zero) and store.
__device__ __forceinline__ void add_store_row(__nv_bfloat16* dst, const float* v, bool has) {
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
        float o[8];
        if (has) {
            const uint4 old = *reinterpret_cast<const uint4*>(dst + 8 * ch);
            unpack8(old.x, old.y, old.z, old.w, o);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = 0.0f;
        }
        uint4 w;
        w.x = pack_bf16(o[0] + v[8 * ch], o[1] + v[8 * ch + 1]);
        w.y = pack_bf16(o[2] + v[8 * ch + 2], o[3] + v[8 * ch + 3]);
        w.z = pack_bf16(o[4] + v[8 * ch + 4], o[5] + v[8 * ch + 5]);
        w.w = pack_bf16(o[6] + v[8 * ch + 6], o[7] + v[8 * ch + 7]);
        *reinterpret_cast<uint4*>(dst + 8 * ch) = w;
    }
}

// The same with the bf16 row already loaded (requested early, so its latency is hidden).
__device__ __forceinline__ void add_store_loaded(__nv_bfloat16* dst, const float* v,
                                                 const uint4 (&old)[4]) {
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
        float o[8];
        unpack8(old[ch].x, old[ch].y, old[ch].z, old[ch].w, o);
        uint4 w;
        w.x = pack_bf16(o[0] + v[8 * ch], o[1] + v[8 * ch + 1]);
        w.y = pack_bf16(o[2] + v[8 * ch + 2], o[3] + v[8 * ch + 3]);
        w.z = pack_bf16(o[4] + v[8 * ch + 4], o[5] + v[8 * ch + 5]);
        w.w = pack_bf16(o[6] + v[8 * ch + 6], o[7] + v[8 * ch + 7]);
        *reinterpret_cast<uint4*>(dst + 8 * ch) = w;
    }
}

// ---------------------------------------------------------------------------------------
// dk, dv window parts: keys [j0, j0 + 128) against the query tiles that can see them.
constexpr uint32_t aK = 0, aV = 32768, aQ = 65536, aD = 131072, aRow = 196608,
                   aBars = aRow + 2048;
constexpr uint32_t kSmemKV = aBars + (uint32_t)sizeof(Bars) + 1024;
static_assert(kSmemKV <= 232448, "shared memory budget");
// TMEM: S^T [0,128) (P^T in its first 64 columns), dP^T [128,256) (dS^T likewise),
// dV [256,384), dK [384,512)
constexpr uint32_t cST = 0, cDPT = 128, cDV = 256, cDK = 384;

__global__ void __launch_bounds__(NT, 1)
    bwd_win_kv_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmD,
                  const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  Plan p, BwdArgs a, const float* rows) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    Bars& S = *reinterpret_cast<Bars*>(sm + aBars);
    float* slse = reinterpret_cast<float*>(sm + aRow);  // [2][128] per query row
    float* sdel = slse + 256;                            // [2][128]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, part = warp >> 2;
    const int row = 32 * quad + lane;  // key of the tile
    const int64_t unit = blockIdx.y, b = unit / p.Hkv, kv = unit % p.Hkv;
    const int64_t j0 = (int64_t)blockIdx.x * 128;
    const int64_t nc = (p.L + CT - 1) / CT;
    const int64_t c_first = j0 / CT;
    const int64_t c_last = min64(nc - 1, (j0 + 127 + WIN - 1) / CT);
    const int nq = (int)(c_last - c_first + 1);
    const int64_t nrow = p.B * p.L * p.Hq;
    WsHeader* hdr = (WsHeader*)a.ws;
    const uint32_t lane_off = (uint32_t)(32 * quad) << 16;

    if (warp == 0) {
        tmem_alloc(&S.tmem, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&S.bar_kv, 1);
        mbar_init(&S.bar_in[0], 1);
        mbar_init(&S.bar_in[1], 1);
        mbar_init(&S.bar_s, 1);
        mbar_init(&S.bar_o, 1);
        mbar_init(&S.bar_fin, 1);
        fence_mbar_init();
        S.abort = 0;
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = S.tmem;
    bool mma_out = false;
    uint64_t* tbar = nullptr;  // a copy phase this thread issued and nobody has waited for
    uint32_t tph = 0;
    if (tid == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmD);
        mbar_arrive_expect_tx(&S.bar_kv, 2 * kTile);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_4d(sm + aK + kb * 16384, &tmK, &S.bar_kv, 64 * kb, (int)kv, (int)j0, (int)b);
            tma_load_4d(sm + aV + kb * 16384, &tmV, &S.bar_kv, 64 * kb, (int)kv, (int)j0, (int)b);
        }
        load_qdy(sm + aQ, sm + aD, &tmQ, &tmD, &S.bar_in[0], kv, c_first, b);
        tbar = &S.bar_in[0];
    }
    const uint64_t dK = kdesc(base + aK), dV = kdesc(base + aV);
    uint32_t ph_in[2] = {0, 0}, ph_s = 0, ph_o = 0;
    bool ok = all_wait(&S.bar_kv, 0, S, hdr, 30);
    const float s2 = p.scale * kLog2e;

    // lse and delta of tile n's rows (the columns of S^T), requested one tile ahead
    float nls = 0.0f, ndl = 0.0f;
    auto row_vals = [&](int64_t cc) {
        const int64_t i = cc * CT + (tid >> 2);
        const int64_t idx = (b * p.L + i) * p.Hq + kv * GQ + (tid & 3);
        nls = i < p.L ? a.lse[idx] : 0.0f;
        ndl = i < p.L ? rows[nrow + idx] : 0.0f;
    };
    if (tid < 128 && nq > 0) row_vals(c_first);

    for (int n = 0; ok && n < nq; ++n) {
        const int buf = n & 1;
        const int64_t c = c_first + n, q0 = c * CT;
        if (tid < 128) {
            slse[buf * 128 + tid] = nls * kLog2e;
            sdel[buf * 128 + tid] = ndl;
            if (n + 1 < nq) row_vals(c + 1);
        }
        ok = all_wait(&S.bar_in[buf], ph_in[buf], S, hdr, 31);
        if (!ok) break;
        ph_in[buf] ^= 1u;
        const uint32_t q_s = base + aQ + buf * kTile, d_s = base + aD + buf * kTile;
        if (tid == 0) {
            tc_fence_after();
            const uint64_t dQ = kdesc(q_s), dD = kdesc(d_s);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t off = ((j >> 2) * 16384 + (j & 3) * 32) >> 4;
                mma_bf16(tb + cST, dK + off, dQ + off, idesc_bf16(128, 128, false, false), j > 0);
                mma_bf16(tb + cDPT, dV + off, dD + off, idesc_bf16(128, 128, false, false), j > 0);
            }
            mma_commit(&S.bar_s);
            mma_out = true;
            // the other buffer's last readers (the previous tile's dV, dK MMAs) are done
            if (n + 1 < nq) {
                load_qdy(sm + aQ + (buf ^ 1) * kTile, sm + aD + (buf ^ 1) * kTile, &tmQ, &tmD,
                         &S.bar_in[buf ^ 1], kv, c + 1, b);
                tbar = &S.bar_in[buf ^ 1];
                tph = ph_in[buf ^ 1];
            }
        }
        ok = all_wait(&S.bar_s, ph_s, S, hdr, 32);
        if (!ok) break;
        ph_s ^= 1u;
        tc_fence_after();
        // P^T and dS^T for key `row`, query rows [32 part, 32 part + 32)
        uint32_t pw[16], dw[16];
        {
            float sv[32], dp[32];
            tmem_ld32(tb + lane_off + cST + 32 * part, sv);
            tmem_ld32(tb + lane_off + cDPT + 32 * part, dp);
            tmem_wait_ld();
            const int64_t j = j0 + row;
            const float* ls = slse + buf * 128 + 32 * part;
            const float* dl = sdel + buf * 128 + 32 * part;
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
                float pv[2], dv2[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = 32 * part + k + e;
                    const int64_t i = q0 + (r >> 2);
                    const bool valid = i < p.L && j <= i && i < j + WIN;
                    pv[e] = valid ? ex2f(fmaf(sv[k + e], s2, -ls[k + e])) : 0.0f;
                    dv2[e] = pv[e] * (dp[k + e] - dl[k + e]) * p.scale;
                }
                pw[k / 2] = pack_bf16(pv[0], pv[1]);
                dw[k / 2] = pack_bf16(dv2[0], dv2[1]);
            }
        }
        tc_fence_before();
        quad_sync(quad);  // every part of this quad has read its S^T, dP^T columns
        tc_fence_after();
        tmem_st16(tb + lane_off + cST + 16 * part, pw);
        tmem_st16(tb + lane_off + cDPT + 16 * part, dw);
        tmem_wait_st();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            // dV += P^T dY, dK += dS^T Q (A from TMEM, 16 query rows per K step)
            const uint64_t dQm = mndesc(q_s, 16384), dDm = mndesc(d_s, 16384);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t acc = (n > 0 || j > 0) ? 1u : 0u;
                mma_bf16_ts(tb + cDV, tb + cST + 8 * j, dDm + ((j * 2048) >> 4),
                            idesc_bf16(128, 128, false, true), acc);
                mma_bf16_ts(tb + cDK, tb + cDPT + 8 * j, dQm + ((j * 2048) >> 4),
                            idesc_bf16(128, 128, false, true), acc);
            }
            mma_commit(&S.bar_o);
        }
        ok = all_wait(&S.bar_o, ph_o, S, hdr, 33);
        if (!ok) break;
        ph_o ^= 1u;
        if (tid == 0) mma_out = false;
        tc_fence_after();
    }

    if (ok) {
        // add the window parts to the state parts (keys j with j + w < L have them)
        const int64_t j = j0 + row;
        float v[32];
        tmem_ld32(tb + lane_off + cDK + 32 * part, v);
        tmem_wait_ld();
        if (j < p.L) {
            const bool has = j + p.w < p.L;
            __nv_bfloat16* dk = (__nv_bfloat16*)a.dk + ((b * p.L + j) * p.Hkv + kv) * DH + 32 * part;
            add_store_row(dk, v, has);
        }
        tmem_ld32(tb + lane_off + cDV + 32 * part, v);
        tmem_wait_ld();
        if (j < p.L) {
            const bool has = j + p.w < p.L;
            __nv_bfloat16* dv = (__nv_bfloat16*)a.dv + ((b * p.L + j) * p.Hkv + kv) * DH + 32 * part;
            add_store_row(dv, v, has);
        }
    } else if (tid == 0) {
        // the pending copy phase, if any, is the one nobody waited for
        const bool pending = tbar != nullptr && !mbar_try_wait(tbar, tph);
        drain(S, mma_out, pending ? tbar : nullptr, tph);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 512);
    }
}

// ---------------------------------------------------------------------------------------
// dq window part: query tiles of a 128-token block against the keys that can reach them.
// The key tile holds the 224 keys from 64 before the block to 32 after it; query tile n
// (tokens [32 n, 32 n + 32) of the block) sees key rows [32 n, 32 n + 128) of it (its own
// chunk, the two before it and, all masked, the one after).
constexpr int KR = 224;                  // key rows staged per block
constexpr uint32_t kHalfK = KR * 128;    // bytes of one 64-column half of the key tile
constexpr uint32_t bK = 0, bV = 2 * kHalfK, bQ = 4 * kHalfK, bD = bQ + kTile, bBars = bD + kTile;
constexpr uint32_t kSmemQ = bBars + (uint32_t)sizeof(Bars) + 1024;
static_assert(kSmemQ <= 232448, "shared memory budget");
// TMEM: S [0,128) (dS in its first 64 columns), dP [128,256), dQ [256,384)
constexpr uint32_t cS = 0, cDP = 128, cDQ = 256;

__global__ void __launch_bounds__(NT, 1)
    bwd_win_q_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmD,
                 const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 Plan p, BwdArgs a, const float* rows) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    Bars& S = *reinterpret_cast<Bars*>(sm + bBars);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, part = warp >> 2;
    const int row = 32 * quad + lane;  // query row of the tile: 4 token + head
    const int64_t unit = blockIdx.y, b = unit / p.Hkv, kv = unit % p.Hkv;
    const int64_t c0 = (int64_t)blockIdx.x * 4;
    const int64_t nc = (p.L + CT - 1) / CT;
    const int nq = (int)min64(4, nc - c0);
    const int64_t nrow = p.B * p.L * p.Hq;
    WsHeader* hdr = (WsHeader*)a.ws;
    const uint32_t lane_off = (uint32_t)(32 * quad) << 16;

    if (warp == 0) {
        tmem_alloc(&S.tmem, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&S.bar_kv, 1);
        mbar_init(&S.bar_in[0], 1);
        mbar_init(&S.bar_s, 1);
        mbar_init(&S.bar_o, 1);
        mbar_init(&S.bar_fin, 1);
        fence_mbar_init();
        S.abort = 0;
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = S.tmem;
    bool mma_out = false;
    uint64_t* tbar = nullptr;
    uint32_t tph = 0;
    if (tid == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmD);
        // keys from 64 before the block (zero-filled before the sequence start)
        mbar_arrive_expect_tx(&S.bar_kv, 4 * kHalfK);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_4d(sm + bK + kb * kHalfK, &tmK, &S.bar_kv, 64 * kb, (int)kv,
                        (int)(c0 * CT - WIN), (int)b);
            tma_load_4d(sm + bV + kb * kHalfK, &tmV, &S.bar_kv, 64 * kb, (int)kv,
                        (int)(c0 * CT - WIN), (int)b);
        }
        load_qdy(sm + bQ, sm + bD, &tmQ, &tmD, &S.bar_in[0], kv, c0, b);
        tbar = &S.bar_in[0];
    }
    uint32_t ph_in = 0, ph_s = 0, ph_o = 0;
    bool ok = all_wait(&S.bar_kv, 0, S, hdr, 40);
    const float s2 = p.scale * kLog2e;
    const uint64_t dQ = kdesc(base + bQ), dD = kdesc(base + bD);

    // this thread's row: lse and delta requested one tile ahead, the dq row (holding the
    // state part) at the top of its tile; both are used late in the tile
    float nls = 0.0f, ndl = 0.0f;
    auto row_vals = [&](int64_t cc) {
        const int64_t i = cc * CT + (row >> 2);
        const int64_t idx = (b * p.L + i) * p.Hq + kv * GQ + (row & 3);
        nls = i < p.L ? a.lse[idx] : 0.0f;
        ndl = i < p.L ? rows[nrow + idx] : 0.0f;
    };
    if (nq > 0) row_vals(c0);

    for (int n = 0; ok && n < nq; ++n) {
        const int64_t c = c0 + n, q0 = c * CT;
        const float ls = nls * kLog2e, dl = ndl;
        if (n + 1 < nq) row_vals(c + 1);
        uint4 oldq[4];
        {
            const int64_t i = q0 + (row >> 2);
            const int64_t idx = (b * p.L + i) * p.Hq + kv * GQ + (row & 3);
            const uint4* src = reinterpret_cast<const uint4*>((const __nv_bfloat16*)a.dq + idx * DH + 32 * part);
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) oldq[ch] = i < p.L ? src[ch] : make_uint4(0u, 0u, 0u, 0u);
        }
        ok = all_wait(&S.bar_in[0], ph_in, S, hdr, 41);
        if (!ok) break;
        ph_in ^= 1u;
        if (tid == 0) {
            tc_fence_after();
            const uint64_t dKn = kdesc(base + bK + n * 4096), dVn = kdesc(base + bV + n * 4096);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t qo = ((j >> 2) * 16384 + (j & 3) * 32) >> 4;
                const uint32_t ko = ((j >> 2) * kHalfK + (j & 3) * 32) >> 4;
                mma_bf16(tb + cS, dQ + qo, dKn + ko, idesc_bf16(128, 128, false, false), j > 0);
                mma_bf16(tb + cDP, dD + qo, dVn + ko, idesc_bf16(128, 128, false, false), j > 0);
            }
            mma_commit(&S.bar_s);
            mma_out = true;
        }
        ok = all_wait(&S.bar_s, ph_s, S, hdr, 42);
        if (!ok) break;
        ph_s ^= 1u;
        tc_fence_after();
        // the query and dy tiles are consumed: the next tile's copies start now
        if (tid == 0 && n + 1 < nq) {
            load_qdy(sm + bQ, sm + bD, &tmQ, &tmD, &S.bar_in[0], kv, c + 1, b);
            tbar = &S.bar_in[0];
            tph = ph_in;
        }
        // dS for query row `row` against keys of chunk c - 2 + part
        const int64_t i = q0 + (row >> 2);
        const int64_t idx = (b * p.L + i) * p.Hq + kv * GQ + (row & 3);
        const bool rv = i < p.L;
        uint32_t dw[16];
        {
            const int64_t kbase = (c - 2 + part) * CT;
            // keys kbase + u with i - w < key <= i and key >= 0
            const int64_t lo = max64(max64(0, i - WIN + 1 - kbase), -kbase);
            const int64_t hi = min64(31, i - kbase);
            uint32_t vm = 0;
            if (rv && part < 3 && hi >= lo)
                vm = (uint32_t)(((2ull << hi) - 1ull) & ~((1ull << lo) - 1ull));
            if (part < 3) {  // the same for the whole warp: TMEM loads are warp-wide
                float sv[32], dp[32];
                tmem_ld32(tb + lane_off + cS + 32 * part, sv);
                tmem_ld32(tb + lane_off + cDP + 32 * part, dp);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 32; k += 2) {
                    float d2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float pv =
                            ((vm >> (k + e)) & 1u) ? ex2f(fmaf(sv[k + e], s2, -ls)) : 0.0f;
                        d2[e] = pv * (dp[k + e] - dl) * p.scale;
                    }
                    dw[k / 2] = pack_bf16(d2[0], d2[1]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) dw[e] = 0u;
            }
        }
        tc_fence_before();
        quad_sync(quad);
        tc_fence_after();
        tmem_st16(tb + lane_off + cS + 16 * part, dw);
        tmem_wait_st();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            // dQ = dS K over the three chunks that hold window keys (the fourth is masked)
            const uint64_t dKm = mndesc(base + bK + n * 4096, kHalfK);
#pragma unroll
            for (int j = 0; j < 6; ++j)
                mma_bf16_ts(tb + cDQ, tb + cS + 8 * j, dKm + ((j * 2048) >> 4),
                            idesc_bf16(128, 128, false, true), j > 0);
            mma_commit(&S.bar_o);
        }
        ok = all_wait(&S.bar_o, ph_o, S, hdr, 43);
        if (!ok) break;
        ph_o ^= 1u;
        if (tid == 0) mma_out = false;
        tc_fence_after();
        // dq += window part (columns [32 part, 32 part + 32) of this row)
        float v[32];
        tmem_ld32(tb + lane_off + cDQ + 32 * part, v);
        tmem_wait_ld();
        if (rv) add_store_loaded((__nv_bfloat16*)a.dq + idx * DH + 32 * part, v, oldq);
        tc_fence_before();
        __syncthreads();  // S, dP, dQ columns are free for the next tile
    }

    if (!ok && tid == 0) {
        const bool pending = tbar != nullptr && !mbar_try_wait(tbar, tph);
        drain(S, mma_out, pending ? tbar : nullptr, tph);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 512);
    }
}

// ---------------------------------------------------------------------------------------
// Reverse segment pass: what a segment adds to the state adjoint at its start,
//   [dH | dz] = sum_i e^{b_i} (.) phi(q_i) a_i [dy_i, -delta_i]
// (b_i = cumulative log-sigmoid gate from the segment start to token i), and its total
// log-decay, walking the segment backwards in 32-token steps of 128 query rows.  The
// weighted feature rows q^ = phi(q) e^{b} a form the A operand (features are the MMA rows)
// of dH += q^^T dY.
constexpr uint32_t rQ = 0, rD = 32768, rQh = 65536, rW = 98304, rG = 114688,
                   rE = rG + 8192;                 // e^{b_t} fp32 [32][EPR]
constexpr int EPR = 132;                           // padded row pitch (floats) of the decay table
constexpr uint32_t rX = rE + 32 * EPR * 4;         // exchanges [4][128] x 4, -delta [128]
constexpr uint32_t rBars = rX + 9216;
struct RSmall {
    uint64_t bar_q, bar_d, bar_g, bar_u, bar_h, bar_fin;
    uint32_t tmem;
    volatile int abort;
    float dz[128], el[128];
};
constexpr uint32_t rQl = 151552;                    // low bf16 part of q^ (same layout)
static_assert(rBars + sizeof(RSmall) <= rQl, "reverse-pass layout");
constexpr uint32_t kSmemRev = rQl + 32768 + 1024;
static_assert(kSmemRev <= 232448, "shared memory budget");

__device__ __forceinline__ bool rev_wait(uint64_t* bar, uint32_t& ph, RSmall& S, WsHeader* hdr,
                                         unsigned where) {
    bool fail = false;
    if (!mbar_try_wait(bar, ph)) {
        const long long t0 = clock64();
        while (!mbar_try_wait(bar, ph)) {
            if (S.abort || clock64() - t0 > kTimeout) {
                fail = true;
                break;
            }
        }
    }
    if (fail && !S.abort) {
        S.abort = 1;
        report(hdr, LIZARD_ERR_TIMEOUT, where);
    }
    if (!fail) ph ^= 1u;
    return !__syncthreads_or(fail);
}

__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* tm, uint64_t* bar,
                                          int64_t kv, int64_t c, int64_t b) {
    mbar_arrive_expect_tx(bar, kTile);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb)
        tma_load_4d(dst + kb * 16384, tm, bar, 64 * kb, (int)(kv * GQ), (int)(c * CT), (int)b);
}

__device__ __forceinline__ float log_sigmoid_f(float x) {
    return fminf(x, 0.0f) - __logf(1.0f + __expf(-fabsf(x)));
}

__global__ void __launch_bounds__(NT, 1)
    bwd_rev_local_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmD,
                     const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmG,
                     Plan p, BwdArgs a, const float* rows, float* rev_rec) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    RSmall& S = *reinterpret_cast<RSmall*>(sm + rBars);
    float* xum = reinterpret_cast<float*>(sm + rX);  // [4][128]
    float* xus = xum + 512;                          // [4][128]
    float* gpart = xum + 1024;                       // [4][128]
    float* zq = xum + 1536;                          // [4][128]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, part = warp >> 2;
    const int row = 32 * quad + lane;
    const int64_t unit = blockIdx.x, seg = blockIdx.y + 1;
    const int64_t b = unit / p.Hkv, kv = unit % p.Hkv;
    const int64_t U = p.B * p.Hkv;
    const int64_t s0 = seg * p.seg_len, s1 = min64(p.L, s0 + p.seg_len);
    const int64_t c_first = s0 / CT, c_last = (s1 - 1) / CT;
    const int64_t nrow = p.B * p.L * p.Hq;
    WsHeader* hdr = (WsHeader*)a.ws;
    const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
    constexpr uint32_t cH = 0, cU = 128;

    if (warp == 0) {
        tmem_alloc(&S.tmem, 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&S.bar_q, 1);
        mbar_init(&S.bar_d, 1);
        mbar_init(&S.bar_g, 1);
        mbar_init(&S.bar_u, 1);
        mbar_init(&S.bar_h, 1);
        mbar_init(&S.bar_fin, 1);
        fence_mbar_init();
        S.abort = 0;
    }
    if (tid < 128) S.dz[tid] = 0.0f;
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = S.tmem;
    {
        float v[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = 0.0f;
        tmem_st32(tb + lane_off + cH + 32 * part, v);
        tmem_wait_st();
    }
    bool q_out = false, d_out = false, g_out = false, mma_out = false;
    if (tid == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmD);
        prefetch_tmap(&tmG);
        mbar_arrive_expect_tx(&S.bar_q, kTile + 16384u);
        tma_load_3d(sm + rW, &tmW, &S.bar_q, 0, 0, (int)kv);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
            tma_load_4d(sm + rQ + kb * 16384, &tmQ, &S.bar_q, 64 * kb, (int)(kv * GQ),
                        (int)(c_last * CT), (int)b);
        load_tile(sm + rD, &tmD, &S.bar_d, kv, c_last, b);
        mbar_arrive_expect_tx(&S.bar_g, 8192u);
        tma_load_4d(sm + rG, &tmG, &S.bar_g, 0, (int)kv, (int)(c_last * CT), (int)b);
        q_out = d_out = g_out = true;
    }
    tc_fence_before();
    __syncthreads();
    const uint64_t dQ = kdesc(base + rQ), dW = mndesc(base + rW, 16384);
    const uint64_t dQh = mndesc(base + rQh, 16384), dD = mndesc(base + rD, 16384),
                   dQl = mndesc(base + rQl, 16384);
    uint32_t ph_q = 0, ph_d = 0, ph_g = 0, ph_u = 0, ph_h = 0;
    float lam_tot = 0.0f;
    bool ok = true;

    for (int64_t c = c_last; c >= c_first; --c) {
        const int64_t q0 = c * CT;
        const int n = (int)min64(CT, s1 - q0);
        const bool more = c > c_first;
        // (1) U_q = q Wf
        ok = rev_wait(&S.bar_q, ph_q, S, hdr, 50);
        if (!ok) break;
        if (tid == 0) {
            q_out = false;
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t off = ((j >> 2) * 16384 + (j & 3) * 32) >> 4;
                mma_bf16(tb + cU, dQ + off, dW + ((j * 2048) >> 4), idesc_bf16(128, 64, false, true),
                         j > 0);
            }
            mma_commit(&S.bar_u);
            mma_out = true;
        }
        // (2) gates: e^{b_t} per token and feature (at most 1), e^{b_31} for the decay
        ok = rev_wait(&S.bar_g, ph_g, S, hdr, 51);
        if (!ok) break;
        {
            const int gf = tid & 127, gq = tid >> 7;
            // e^{b_t} = prod_{s <= t} Gamma_s with Gamma = 1 / (1 + e^{-g}): prefix products
            // inside the thread's quarter times the earlier quarters' products; the step's
            // log-decay (for the records) from the quarter products renormalised every 4
            // tokens, one logarithm per thread
            const __nv_bfloat16* sg = (const __nv_bfloat16*)(sm + rG);
            float pre[8];
            float pp = 1.0f, mq = 1.0f;
            int eq = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int tt = 8 * gq + j;
                const float gam =
                    tt < n ? rcpf(1.0f + ex2f(-__bfloat162float(sg[tt * 128 + gf]) * kLog2e)) : 1.0f;
                pp *= gam;
                pre[j] = pp;
                mq *= gam;
                if ((j & 3) == 3) {
                    int e;
                    mq = frexpf(mq, &e);
                    eq += e;
                }
            }
            gpart[gq * 128 + gf] = pp;
            zq[gq * 128 + gf] = (__log2f(mq) + (float)eq) * kLn2;
            __syncthreads();
            const float q0 = gpart[gf], q1 = gpart[128 + gf], q2 = gpart[256 + gf];
            const float before = gq == 0 ? 1.0f : gq == 1 ? q0 : gq == 2 ? q0 * q1 : (q0 * q1) * q2;
            // kept in fp32: the adjoint records feed the gate gradient, a difference of two
            // nearly equal sums that bf16 weights would not cancel consistently
            float* Eb = (float*)(sm + rE);
#pragma unroll
            for (int j = 0; j < 8; ++j) Eb[(8 * gq + j) * EPR + gf] = pre[j] * before;
            if (gq == 0) {
                S.el[gf] = ((q0 * q1) * q2) * gpart[384 + gf];
                lam_tot += (zq[gf] + zq[128 + gf]) + (zq[256 + gf] + zq[384 + gf]);
            }
        }
        __syncthreads();
        if (tid == 0) {
            g_out = false;
            if (more) {
                mbar_arrive_expect_tx(&S.bar_g, 8192u);
                tma_load_4d(sm + rG, &tmG, &S.bar_g, 0, (int)kv, (int)((c - 1) * CT), (int)b);
                g_out = true;
            }
        }
        // (3) the adjoint from later steps decays over this step: dH, dz *= e^{b_31}
        {
            float v[32];
            tmem_ld32(tb + lane_off + cH + 32 * part, v);
            tmem_wait_ld();
            const float el = S.el[row];
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] *= el;
            tmem_st32(tb + lane_off + cH + 32 * part, v);
            tmem_wait_st();
        }
        // (4) q^ = phi(q) e^{b_t} a for row = 4 t + head
        ok = rev_wait(&S.bar_u, ph_u, S, hdr, 52);
        if (!ok) break;
        tc_fence_after();
        if (tid == 0) {
            mma_out = false;
            if (more) {
                mbar_arrive_expect_tx(&S.bar_q, kTile);
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
                    tma_load_4d(sm + rQ + kb * 16384, &tmQ, &S.bar_q, 64 * kb, (int)(kv * GQ),
                                (int)((c - 1) * CT), (int)b);
                q_out = true;
            }
        }
        {
            const int t = row >> 2, sib = part ^ 1;
            const int64_t i = q0 + t;
            const int64_t idx = (b * p.L + i) * p.Hq + kv * GQ + (row & 3);
            const float ar = t < n ? rows[idx] : 0.0f;
            if (part == 0) zq[512 + row] = t < n ? -rows[nrow + idx] : 0.0f;  // -delta per row
            float uv[32];
            tmem_ld32(tb + lane_off + cU + 32 * (part & 1), uv);
            tmem_wait_ld();
            float uext = -INFINITY;
            if (part < 2) {
#pragma unroll
                for (int k = 0; k < 32; ++k) uext = fmaxf(uext, uv[k]);
            } else {
#pragma unroll
                for (int k = 0; k < 32; ++k) uext = fmaxf(uext, -uv[k]);
            }
            xum[part * 128 + row] = uext;
            quad_sync(quad);
            const float f2 = part < 2 ? kLog2e : -kLog2e;
            const float cst = -fmaxf(xum[part * 128 + row], xum[sib * 128 + row]) * kLog2e;
            float usum = 0.0f;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                uv[k] = ex2f(fmaf(uv[k], f2, cst));
                usum += uv[k];
            }
            xus[part * 128 + row] = usum;
            quad_sync(quad);
            const float sc = ar / (xus[part * 128 + row] + xus[sib * 128 + row]);
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                const int f0 = 32 * part + 8 * ch;
                const float4* ep = reinterpret_cast<const float4*>(sm + rE + (size_t)(t * EPR + f0) * 4u);
                const float4 e0 = ep[0], e1 = ep[1];
                const float eb[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
                float qh[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) qh[e] = uv[8 * ch + e] * sc * eb[e];
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) split2(qh[2 * e], qh[2 * e + 1], hi[e], lo[e]);
                const uint32_t o = (part >> 1) * 16384 + sw128(row, 4 * (part & 1) + ch);
                st_shared_v4(base + rQh + o, hi[0], hi[1], hi[2], hi[3]);
                st_shared_v4(base + rQl + o, lo[0], lo[1], lo[2], lo[3]);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // (5) dH += q^^T dY on the tensor cores while the threads sum dz
        if (tid == 0) {
            if (!mbar_wait(&S.bar_d, ph_d, kTimeout)) {
                S.abort = 1;
                report(hdr, LIZARD_ERR_TIMEOUT, 53);
            } else {
                ph_d ^= 1u;
                d_out = false;
                tc_fence_after();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    mma_bf16(tb + cH, dQh + ((j * 2048) >> 4), dD + ((j * 2048) >> 4),
                             idesc_bf16(128, 128, true, true), 1);
                    mma_bf16(tb + cH, dQl + ((j * 2048) >> 4), dD + ((j * 2048) >> 4),
                             idesc_bf16(128, 128, true, true), 1);
                }
                mma_commit(&S.bar_h);
                mma_out = true;
            }
        }
        {
            // dz_f += sum_rows q^[row][f] (-delta_row), from the bf16 tile the MMA reads
            const int f = tid & 127, gq = tid >> 7;
            const __nv_bfloat16* qh = (const __nv_bfloat16*)(sm + rQh);
            const __nv_bfloat16* ql = (const __nv_bfloat16*)(sm + rQl);
            float zs[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // four chains: the loads overlap
#pragma unroll
            for (int r = 32 * gq; r < 32 * gq + 32; ++r) {
                const uint32_t off = ((f >> 6) * 16384 + sw128(r, (f & 63) >> 3) + (f & 7) * 2) / 2;
                zs[r & 3] = fmaf(__bfloat162float(qh[off]) + __bfloat162float(ql[off]), zq[512 + r], zs[r & 3]);
            }
            zq[gq * 128 + f] = (zs[0] + zs[1]) + (zs[2] + zs[3]);
        }
        __syncthreads();
        if (tid < 128)
            S.dz[tid] = fmaf(S.el[tid], S.dz[tid], (zq[tid] + zq[128 + tid]) + (zq[256 + tid] + zq[384 + tid]));
        ok = rev_wait(&S.bar_h, ph_h, S, hdr, 54);
        if (!ok) break;
        tc_fence_after();
        if (tid == 0) {
            mma_out = false;
            if (more) {
                load_tile(sm + rD, &tmD, &S.bar_d, kv, c - 1, b);
                d_out = true;
            }
        }
    }

    if (ok) {
        float* r = rev_rec + ((size_t)seg * (size_t)U + (size_t)unit) * p.rec_floats;
        float v[32];
        tmem_ld32(tb + lane_off + cH + 32 * part, v);
        tmem_wait_ld();
        // through the (now idle) q and dY tiles, then coalesced to the record
        staged_row_write(sm + rQ, row, part, v);
        __syncthreads();
        stage_record_out(r, sm + rQ);
        if (tid < 128) {
            r[128 * DH + tid] = S.dz[tid];
            r[128 * DH + 128 + tid] = lam_tot;
        }
    } else if (tid == 0) {
        if (mma_out) {
            mma_commit(&S.bar_fin);
            mbar_wait(&S.bar_fin, 0, kTimeout);
        }
        if (q_out) mbar_wait(&S.bar_q, ph_q, kTimeout);
        if (g_out) mbar_wait(&S.bar_g, ph_g, kTimeout);
        if (d_out) mbar_wait(&S.bar_d, ph_d, kTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 256);
    }
}

// ---------------------------------------------------------------------------------------
// Forward-direction walk of the backward on the tensor cores: the state part of dq, the
// phi(q)-side of dB, the dWf and dt partials of a segment, walking it in 32-token steps of
// 128 query rows (row = 4 token + head) with the forward's state recurrence.  With
// a_i = e^{-lse_i}, delta_i = dy_i . y_i and the forward's decay reference r of a step:
//   D    = dY (e^{r} (.) H)^T + c k~i            c_it = dy_i . v'_t - delta_i,  t <= i
//   dphi(q)_i = a_i e^{b_i - r} (.) (D_i - delta_i e^{r} (.) z)
//   du   = phi+ (.) (dphi+ - phi+ . dphi+) - phi- (.) (dphi- - phi- . dphi-)
//   dq   = du Wf^T,   dWf += q^T du,   dB_i += sum_heads phi(q_i) (.) dphi(q_i)
// and the state moves on as in the forward: H <- e^{b_31} (.) H + k~u^T V_d.
// dB feeds a reverse cumulative sum whose terms nearly cancel, so the operands of D that
// are not exact in bf16 (the state copy, c, k~i) go in as a high and a low bf16 part, and
// the decay factors stay in fp32.  Each thread owns 16 u-values of its row and both
// feature-map halves built from them, so the feature-map backward needs no exchange of
// feature values.
constexpr uint32_t wQ = 0, wD = 32768, wK = 65536, wV = 73728, wW = 81920, wHh = 98304,
                   wHl = 131072, wKih = 163840, wKil = 172032, wKu = 180224, wB = 188416,
                   wG = 204800, wX = 212992, wSm = 217088;
struct WSmall {
    uint64_t bar_tma, bar_u, bar_d1, bar_d2, bar_q, bar_fin;
    uint32_t tmem;
    volatile int abort;
    float z[128], zs[128], cf[128];
    float dts[4][4];
};
constexpr uint32_t kSmemFW = wSm + (uint32_t)sizeof(WSmall) + 1024;
static_assert(kSmemFW <= 232448, "shared memory budget");
// TMEM: H [0,128), D [128,256), U_q [256,320) and U_k [320,384) -> dq [256,384),
// C [384,416) -> du (bf16 pairs) [384,416), c high [416,432), c low [432,448), dWf [448,512)
constexpr uint32_t fH = 0, fD = 128, fUq = 256, fUk = 320, fDQ = 256, fC = 384, fDU = 384,
                   fCh = 416, fCl = 432, fDW = 448;

__device__ __forceinline__ bool fw_wait(uint64_t* bar, uint32_t& ph, WSmall& S, WsHeader* hdr,
                                        unsigned where) {
    bool fail = false;
    if (!mbar_try_wait(bar, ph)) {
        const long long t0 = clock64();
        while (!mbar_try_wait(bar, ph)) {
            if (S.abort || clock64() - t0 > kTimeout) {
                fail = true;
                break;
            }
        }
    }
    if (fail && !S.abort) {
        S.abort = 1;
        report(hdr, LIZARD_ERR_TIMEOUT, where);
    }
    if (!fail) ph ^= 1u;
    return !__syncthreads_or(fail);
}

__device__ __forceinline__ float clamp80f(float x) { return fminf(fmaxf(x, -80.0f), 80.0f); }


// Delayed keys or values of chunk c (two 64-column halves of 32 rows, 4 KB apart).
__device__ __forceinline__ void load_delayed(uint8_t* dst, const CUtensorMap* tm, uint64_t* bar,
                                             int64_t kv, int64_t c, int64_t b) {
#pragma unroll
    for (int kb = 0; kb < 2; ++kb)
        tma_load_4d(dst + kb * 4096, tm, bar, 64 * kb, (int)kv, (int)((c - 2) * CT), (int)b);
}

// KEYF: the masked decay reading (each delayed key enters with its phi scaled by the product
// of the w gates it saw in the window, e^{kd} from a.kdec); a separate instantiation, so the
// other readings' code is not touched by it.
template <bool KEYF>
__global__ void __launch_bounds__(NT, 1)
    bwd_fwalk_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDY,
                 const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmG,
                 const __grid_constant__ CUtensorMap tmDQ, Plan p, BwdArgs a, const float* rows,
                 const float* fwd_rec, float* dB, float* dWp, float* dtp, const int* flags) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    WSmall& S = *reinterpret_cast<WSmall*>(sm + wSm);
    float* xa = reinterpret_cast<float*>(sm + wX);   // [4][128]
    float* xb = xa + 512;                            // [4][128]
    float* suk = reinterpret_cast<float*>(sm + wG);  // staged U_k rows [32][64]
    float* etab = reinterpret_cast<float*>(sm + wB); // e^{b_t - r} [32][128] fp32

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, part = warp >> 2;
    const int row = 32 * quad + lane;
    const int64_t unit = blockIdx.x, seg = blockIdx.y;
    const int64_t b = unit / p.Hkv, kv = unit % p.Hkv;
    const int64_t U = p.B * p.Hkv;
    const int64_t s0 = seg * p.seg_len, s1 = min64(p.L, s0 + p.seg_len);
    const int64_t c_begin = s0 / CT, c_end = (s1 + CT - 1) / CT;
    const int64_t nrow = p.B * p.L * p.Hq;
    WsHeader* hdr = (WsHeader*)a.ws;
    const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
    constexpr uint32_t kStepBytes = 2 * kTile + 8192u + 8192u + 8192u;  // q, dY, k', v', gates
    // a segment whose gates close too hard for the factored decays is the SIMT walk's
    if (flags[seg * U + unit] != 0) return;

    if (warp == 0) {
        tmem_alloc(&S.tmem, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&S.bar_tma, 1);
        mbar_init(&S.bar_u, 1);
        mbar_init(&S.bar_d1, 1);
        mbar_init(&S.bar_d2, 1);
        mbar_init(&S.bar_q, 1);
        mbar_init(&S.bar_fin, 1);
        fence_mbar_init();
        S.abort = 0;
    }
    const float* rec = seg > 0 ? fwd_rec + ((size_t)seg * (size_t)U + (size_t)unit) * p.rec_floats
                               : nullptr;
    if (tid < 128) S.z[tid] = rec ? rec[128 * DH + tid] : 0.0f;
    if (tid < 16) S.dts[tid >> 2][tid & 3] = 0.0f;
    if (rec) stage_record_in(sm + wQ, rec);  // wQ, wD: the first step's copies land there later
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = S.tmem;
    {
        float v[32];
        staged_row_read(sm + wQ, rec != nullptr, row, part, v);
        tmem_st32(tb + lane_off + fH + 32 * part, v);
        tmem_wait_st();
    }
    __syncthreads();  // the staged rows are read before the copies below overwrite them
    bool tma_out = false, mma_out = false;
    if (tid == 0 && c_begin < c_end) {
        fence_async_smem();
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmDY);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmG);
        mbar_arrive_expect_tx(&S.bar_tma, kStepBytes + 16384u);
        tma_load_3d(sm + wW, &tmW, &S.bar_tma, 0, 0, (int)kv);
        load_delayed(sm + wK, &tmK, &S.bar_tma, kv, c_begin, b);
        load_delayed(sm + wV, &tmV, &S.bar_tma, kv, c_begin, b);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_4d(sm + wQ + kb * 16384, &tmQ, &S.bar_tma, 64 * kb, (int)(kv * GQ),
                        (int)(c_begin * CT), (int)b);
            tma_load_4d(sm + wD + kb * 16384, &tmDY, &S.bar_tma, 64 * kb, (int)(kv * GQ),
                        (int)(c_begin * CT), (int)b);
        }
        tma_load_4d(sm + wG, &tmG, &S.bar_tma, 0, (int)kv, (int)(c_begin * CT), (int)b);
        tma_out = true;
    }
    tc_fence_before();
    __syncthreads();
    const uint64_t dQk = kdesc(base + wQ), dDk = kdesc(base + wD), dKk = kdesc(base + wK),
                   dVk = kdesc(base + wV), dHh = kdesc(base + wHh), dHl = kdesc(base + wHl),
                   dWk = kdesc(base + wW);
    const uint64_t dWm = mndesc(base + wW, 16384), dVm = mndesc(base + wV, 4096),
                   dKih = mndesc(base + wKih, 4096), dKil = mndesc(base + wKil, 4096),
                   dKum = mndesc(base + wKu, 4096), dQm = mndesc(base + wQ, 16384),
                   dDUm = mndesc(base + wKih, 16384), dKulm = mndesc(base + wD, 4096);
    uint32_t ph_tma = 0, ph_u = 0, ph_d1 = 0, ph_d2 = 0, ph_q = 0;
    bool ok = true, dw_init = false;
    float dts_acc = 0.0f;

    for (int64_t c = c_begin; c < c_end; ++c) {
        const int64_t t0 = c * CT;
        const int n = (int)min64(CT, s1 - t0);
        if (KEYF && tid < 128) {  // the next step's key factors (32 rows), into L2
            const int64_t tn = t0 + CT + (tid >> 2);
            if (tn - WIN >= 0 && tn < s1)
                prefetch_l2(a.kdec + ((b * p.L + tn - WIN) * p.Hkv + kv) * 128 + 32 * (tid & 3));
        }
        const bool more = c + 1 < c_end;
        ok = fw_wait(&S.bar_tma, ph_tma, S, hdr, 60);
        if (!ok) break;
        if (tid == 0) {
            tma_out = false;
            tc_fence_after();
            // (1) projections: U_k of the delayed keys (rows 0..31 of the tile; the MMA's other
            //     rows read the neighbouring tiles and are never used), U_q
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t koff = ((j >> 2) * 16384 + (j & 3) * 32) >> 4;
                const uint32_t kdoff = ((j >> 2) * 4096 + (j & 3) * 32) >> 4;
                const uint64_t bw = dWm + ((j * 2048) >> 4);
                mma_bf16(tb + fUk, dKk + kdoff, bw, idesc_bf16(128, 64, false, true), j > 0);
                mma_bf16(tb + fUq, dQk + koff, bw, idesc_bf16(128, 64, false, true), j > 0);
            }
            mma_commit(&S.bar_u);
            mma_out = true;
        }
        // (2) gates: cumulative log-sigmoid b (fp32 table), reference r = b_15
        const int gf = tid & 127, gq = tid >> 7;
        {
            const __nv_bfloat16* sg = (const __nv_bfloat16*)(sm + wG);
            float bt[8];
            float run = 0.0f;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const int tt = 8 * gq + t;
                run += tt < n ? log_sigmoid_f(__bfloat162float(sg[tt * 128 + gf])) : 0.0f;
                bt[t] = run;
            }
            xa[gq * 128 + gf] = run;
            // the previous step's dq tile has left the state-copy buffer before phase (3)
            // writes it again (the barrier orders this for every thread)
            if (tid == 0) bulk_wait_read();
            __syncthreads();
            const float g0 = xa[gf], g1 = xa[128 + gf], g2 = xa[256 + gf], g3 = xa[384 + gf];
            const float bref = g0 + g1, blast = bref + g2 + g3;
            const float off = gq == 0 ? 0.0f : gq == 1 ? g0 : gq == 2 ? bref : bref + g2;
            // the decay factors of the step relative to r, once per (token, feature): the four
            // heads of a token and the key-side phase read them from the table
#pragma unroll
            for (int t = 0; t < 8; ++t)
                etab[(8 * gq + t) * 128 + gf] = __expf(clamp80f(bt[t] + off - bref));
            if (gq == 0) {
                S.cf[gf] = __expf(blast - bref);
                S.zs[gf] = __expf(bref) * S.z[gf];
            }
        }
        // (3) state copy e^{r} (.) H as high and low bf16 parts; master decayed by e^{b_31}
        {
            const int f = row;
            const float g0 = xa[f], g1 = xa[128 + f], g2 = xa[256 + f], g3 = xa[384 + f];
            const float er = __expf(g0 + g1), el = __expf(g0 + g1 + g2 + g3);
            const int col = 32 * part;
            float v[32];
            tmem_ld32(tb + lane_off + fH + col, v);
            tmem_wait_ld();
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                const uint32_t off = (col / 64) * 16384 + sw128(f, (col & 63) / 8 + ch);
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    split2(er * v[8 * ch + 2 * e], er * v[8 * ch + 2 * e + 1], hi[e], lo[e]);
                st_shared_v4(base + wHh + off, hi[0], hi[1], hi[2], hi[3]);
                st_shared_v4(base + wHl + off, lo[0], lo[1], lo[2], lo[3]);
            }
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] *= el;
            tmem_st32(tb + lane_off + fH + col, v);
            tmem_wait_st();
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            // (4) D = dY H_s^T (high + low parts), C = dY V_d^T
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t koff = ((j >> 2) * 16384 + (j & 3) * 32) >> 4;
                const uint32_t kdoff = ((j >> 2) * 4096 + (j & 3) * 32) >> 4;
                mma_bf16(tb + fD, dDk + koff, dHh + koff, idesc_bf16(128, 128, false, false), j > 0);
                mma_bf16(tb + fD, dDk + koff, dHl + koff, idesc_bf16(128, 128, false, false), 1);
                mma_bf16(tb + fC, dDk + koff, dVk + kdoff, idesc_bf16(128, 32, false, false), j > 0);
            }
            mma_commit(&S.bar_d1);
        }
        // (5) phi(q): this thread's 16 u-values give features f = 16 part + k of both halves
        ok = fw_wait(&S.bar_u, ph_u, S, hdr, 61);
        if (!ok) break;
        tc_fence_after();
        if (tid == 0 && more) {
            // the delayed-key tile is consumed: the next step's copies start
            mbar_arrive_expect_tx(&S.bar_tma, kStepBytes);
            load_delayed(sm + wK, &tmK, &S.bar_tma, kv, c + 1, b);
            tma_out = true;
        }
        if (quad == 0 && part < 2) {
            float w[32];
            tmem_ld32(tb + lane_off + fUk + 32 * part, w);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; k += 4)
                *reinterpret_cast<float4*>(suk + lane * 64 + 32 * part + k) =
                    make_float4(w[k], w[k + 1], w[k + 2], w[k + 3]);
        }
        float php[16], phn[16];
        {
            float u[16];
            tmem_ld8(tb + lane_off + fUq + 16 * part, u);
            tmem_ld8(tb + lane_off + fUq + 16 * part + 8, u + 8);
            tmem_wait_ld();
            float mx = -INFINITY, mn = -INFINITY;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                mx = fmaxf(mx, u[k]);
                mn = fmaxf(mn, -u[k]);
            }
            xa[part * 128 + row] = mx;
            xb[part * 128 + row] = mn;
            quad_sync(quad);
            mx = fmaxf(fmaxf(xa[row], xa[128 + row]), fmaxf(xa[256 + row], xa[384 + row]));
            mn = fmaxf(fmaxf(xb[row], xb[128 + row]), fmaxf(xb[256 + row], xb[384 + row]));
            float sp = 0.0f, sn = 0.0f;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                php[k] = __expf(u[k] - mx);
                phn[k] = __expf(-u[k] - mn);
                sp += php[k];
                sn += phn[k];
            }
            quad_sync(quad);
            xa[part * 128 + row] = sp;
            xb[part * 128 + row] = sn;
            quad_sync(quad);
            sp = (xa[row] + xa[128 + row]) + (xa[256 + row] + xa[384 + row]);
            sn = (xb[row] + xb[128 + row]) + (xb[256 + row] + xb[384 + row]);
            const float ip = 1.0f / sp, in = 1.0f / sn;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                php[k] *= ip;
                phn[k] *= in;
            }
        }
        __syncthreads();
        // (6) phi of the delayed keys -> k~i = phi e^{r - b_t} (high, low), k~u = k~i e^{b_31 - r}
        //     (high now; the low part goes into the dY tile once D and C have read it)
        uint32_t kul[2][2];
        {
            const int t = tid >> 4, sub = tid & 15;
            const bool dvalid = (t0 + t - WIN >= 0) && (t < n);
            float4 kd4[2] = {};  // the delayed key's own log factor (masked reading)
            if (KEYF && dvalid) {
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
                    kd4[kb] = *reinterpret_cast<const float4*>(
                        a.kdec + ((b * p.L + t0 + t - WIN) * p.Hkv + kv) * 128 + 64 * kb + 4 * sub);
            }
            const float4 u4 = *reinterpret_cast<const float4*>(suk + t * 64 + 4 * sub);
            const float u[4] = {u4.x, u4.y, u4.z, u4.w};
            float mx = fmaxf(fmaxf(u[0], u[1]), fmaxf(u[2], u[3]));
            float mn = fminf(fminf(u[0], u[1]), fminf(u[2], u[3]));
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) {
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            }
            float ep[4], en[4], sp = 0.0f, sn = 0.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                ep[e] = __expf(u[e] - mx);
                en[e] = __expf(mn - u[e]);
                sp += ep[e];
                sn += en[e];
            }
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) {
                sp += __shfl_xor_sync(0xffffffffu, sp, o);
                sn += __shfl_xor_sync(0xffffffffu, sn, o);
            }
            const float ip = dvalid ? 1.0f / sp : 0.0f, in = dvalid ? 1.0f / sn : 0.0f;
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
                const int f0 = 64 * kb + 4 * sub;
                float ki[4], ku[4], kf[4] = {1.0f, 1.0f, 1.0f, 1.0f};
                if (KEYF && dvalid) {
                    kf[0] = __expf(kd4[kb].x);
                    kf[1] = __expf(kd4[kb].y);
                    kf[2] = __expf(kd4[kb].z);
                    kf[3] = __expf(kd4[kb].w);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float ph = (kb == 0 ? ep[e] * ip : en[e] * in) * kf[e];
                    ki[e] = ph * rcpf(etab[t * 128 + f0 + e]);  // e^{r - b_t}
                    ku[e] = ki[e] * S.cf[f0 + e];
                }
                const uint32_t off = kb * 4096 + sw128(t, sub >> 1) + (sub & 1) * 8;
                uint32_t h0, l0, h1, l1;
                split2(ki[0], ki[1], h0, l0);
                split2(ki[2], ki[3], h1, l1);
                asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(base + wKih + off), "r"(h0),
                             "r"(h1)
                             : "memory");
                asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(base + wKil + off), "r"(l0),
                             "r"(l1)
                             : "memory");
                uint32_t uh0, uh1;
                split2(ku[0], ku[1], uh0, kul[kb][0]);
                split2(ku[2], ku[3], uh1, kul[kb][1]);
                asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(base + wKu + off), "r"(uh0),
                             "r"(uh1)
                             : "memory");
            }
        }
        fence_async_smem();
        __syncthreads();
        if (tid == 0 && more) {
            // the gate tile and the staged U_k rows are consumed
            tma_load_4d(sm + wG, &tmG, &S.bar_tma, 0, (int)kv, (int)((c + 1) * CT), (int)b);
        }
        // (7) c_it = C_it - delta_i for delayed keys t <= i (8 keys per part), high and low
        const int ti = row >> 2;
        const int64_t ridx = (b * p.L + t0 + ti) * p.Hq + kv * GQ + (row & 3);
        const bool rv = ti < n;
        const float ar = rv ? rows[ridx] : 0.0f, dl = rv ? rows[nrow + ridx] : 0.0f;
        ok = fw_wait(&S.bar_d1, ph_d1, S, hdr, 62);
        if (!ok) break;
        tc_fence_after();
        {
            // low part of k~u into the consumed dY tile (same layout as the high part)
            const int t = tid >> 4, sub = tid & 15;
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
                const uint32_t off = kb * 4096 + sw128(t, sub >> 1) + (sub & 1) * 8;
                asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(base + wD + off),
                             "r"(kul[kb][0]), "r"(kul[kb][1])
                             : "memory");
            }
        }
        {
            float cv[8];
            tmem_ld8(tb + lane_off + fC + 8 * part, cv);
            tmem_wait_ld();
            uint32_t ch[4], cl[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                float x2[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int t = 8 * part + e + h;
                    const bool valid = rv && t <= ti && (t0 + t - WIN >= 0);
                    x2[h] = valid ? cv[e + h] - dl : 0.0f;
                }
                split2(x2[0], x2[1], ch[e / 2], cl[e / 2]);
            }
            tmem_st4(tb + lane_off + fCh + 4 * part, ch);
            tmem_st4(tb + lane_off + fCl + 4 * part, cl);
            tmem_wait_st();
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            // (8) D += c k~i (high x high, high x low, low x high); H += k~u^T V_d
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint32_t bo = (j * 2048) >> 4;
                mma_bf16_ts(tb + fD, tb + fCh + 8 * j, dKih + bo, idesc_bf16(128, 128, false, true), 1);
                mma_bf16_ts(tb + fD, tb + fCh + 8 * j, dKil + bo, idesc_bf16(128, 128, false, true), 1);
                mma_bf16_ts(tb + fD, tb + fCl + 8 * j, dKih + bo, idesc_bf16(128, 128, false, true), 1);
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                mma_bf16(tb + fH, dKum + ((j * 2048) >> 4), dVm + ((j * 2048) >> 4),
                         idesc_bf16(128, 128, true, true), 1);
                mma_bf16(tb + fH, dKulm + ((j * 2048) >> 4), dVm + ((j * 2048) >> 4),
                         idesc_bf16(128, 128, true, true), 1);
            }
            mma_commit(&S.bar_d2);
        }
        // z <- e^{b_31} z + sum_t k~u_t (high + low parts the MMA reads)
        if (tid < 128) {
            const int f = tid;
            float zsum = 0.0f;
            const __nv_bfloat16* kuh = (const __nv_bfloat16*)(sm + wKu);
            const __nv_bfloat16* kul2 = (const __nv_bfloat16*)(sm + wD);
            for (int t = 0; t < CT; ++t) {
                const uint32_t off = ((f >> 6) * 4096 + sw128(t, (f & 63) >> 3) + (f & 7) * 2) / 2;
                zsum += __bfloat162float(kuh[off]) + __bfloat162float(kul2[off]);
            }
            S.z[f] = fmaf(S.cf[f] * S.zs[f], 1.0f, zsum);
        }
        ok = fw_wait(&S.bar_d2, ph_d2, S, hdr, 63);
        if (!ok) break;
        tc_fence_after();
        if (tid == 0 && more) {
            // the delayed values, dY and the low part of k~u are consumed
            load_delayed(sm + wV, &tmV, &S.bar_tma, kv, c + 1, b);
#pragma unroll
            for (int kb = 0; kb < 2; ++kb)
                tma_load_4d(sm + wD + kb * 16384, &tmDY, &S.bar_tma, 64 * kb, (int)(kv * GQ),
                            (int)((c + 1) * CT), (int)b);
        }
        // (9) dphi(q), the phi(q)-side of dB, du
        {
            float Dp[16], Dn[16];
            tmem_ld8(tb + lane_off + fD + 16 * part, Dp);
            tmem_ld8(tb + lane_off + fD + 16 * part + 8, Dp + 8);
            tmem_ld8(tb + lane_off + fD + 64 + 16 * part, Dn);
            tmem_ld8(tb + lane_off + fD + 64 + 16 * part + 8, Dn + 8);
            tmem_wait_ld();
            const int fp = 16 * part, fn = 64 + 16 * part;
            float spd = 0.0f, snd = 0.0f;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float eqp = etab[ti * 128 + fp + k], eqn = etab[ti * 128 + fn + k];
                Dp[k] = ar * eqp * (Dp[k] - dl * S.zs[fp + k]);  // dphi+
                Dn[k] = ar * eqn * (Dn[k] - dl * S.zs[fn + k]);  // dphi-
                spd = fmaf(php[k], Dp[k], spd);
                snd = fmaf(phn[k], Dn[k], snd);
            }
            // dB over the group's heads: rows 4 t .. 4 t + 3 are lanes of this warp
            {
                float bp[16], bn[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    float x = php[k] * Dp[k], y = phn[k] * Dn[k];
                    x += __shfl_xor_sync(0xffffffffu, x, 1);
                    y += __shfl_xor_sync(0xffffffffu, y, 1);
                    x += __shfl_xor_sync(0xffffffffu, x, 2);
                    y += __shfl_xor_sync(0xffffffffu, y, 2);
                    bp[k] = x;
                    bn[k] = y;
                }
                if ((lane & 3) == 0 && rv) {
                    float* dst = dB + ((b * p.L + t0 + ti) * p.Hkv + kv) * 128;
#pragma unroll
                    for (int k = 0; k < 16; k += 4) {
                        *reinterpret_cast<float4*>(dst + fp + k) =
                            make_float4(bp[k], bp[k + 1], bp[k + 2], bp[k + 3]);
                        *reinterpret_cast<float4*>(dst + fn + k) =
                            make_float4(bn[k], bn[k + 1], bn[k + 2], bn[k + 3]);
                    }
                }
            }
            xa[part * 128 + row] = spd;
            xb[part * 128 + row] = snd;
            quad_sync(quad);
            const float Sp = (xa[row] + xa[128 + row]) + (xa[256 + row] + xa[384 + row]);
            const float Sn = (xb[row] + xb[128 + row]) + (xb[256 + row] + xb[384 + row]);
            uint32_t dw8[8];
#pragma unroll
            for (int k = 0; k < 16; k += 2) {
                float d2[2];
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    d2[h] = php[k + h] * (Dp[k + h] - Sp) - phn[k + h] * (Dn[k + h] - Sn);
                dw8[k / 2] = pack_bf16(d2[0], d2[1]);
            }
            // du as the A operand of dq (TMEM) and the B operand of dWf (shared memory)
            tmem_st8(tb + lane_off + fDU + 8 * part, dw8);
            st_shared_v4(base + wKih + sw128(row, 2 * part), dw8[0], dw8[1], dw8[2], dw8[3]);
            st_shared_v4(base + wKih + sw128(row, 2 * part + 1), dw8[4], dw8[5], dw8[6], dw8[7]);
            tmem_wait_st();
        }
        if (rv) dts_acc = fmaf(ar, dl, dts_acc);  // rows of one head are summed at the end
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            // (10) dq = du Wf^T; dWf += q^T du
#pragma unroll
            for (int j = 0; j < 4; ++j)
                mma_bf16_ts(tb + fDQ, tb + fDU + 8 * j, dWk + ((j * 32) >> 4),
                            idesc_bf16(128, 128, false, false), j > 0);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                mma_bf16(tb + fDW, dQm + ((j * 2048) >> 4), dDUm + ((j * 2048) >> 4),
                         idesc_bf16(128, 64, true, true), (dw_init || j > 0) ? 1u : 0u);
            mma_commit(&S.bar_q);
        }
        dw_init = true;
        ok = fw_wait(&S.bar_q, ph_q, S, hdr, 64);
        if (!ok) break;
        tc_fence_after();
        if (tid == 0) {
            mma_out = false;
            if (more) {
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
                    tma_load_4d(sm + wQ + kb * 16384, &tmQ, &S.bar_tma, 64 * kb, (int)(kv * GQ),
                                (int)((c + 1) * CT), (int)b);
            }
        }
        {
            // the dq tile (state part) through the idle state-copy buffer and one TMA store;
            // rows past the end of the sequence fall outside the tensor and are dropped
            float v[32];
            tmem_ld32(tb + lane_off + fDQ + 32 * part, v);
            tmem_wait_ld();
#pragma unroll
            for (int ch = 0; ch < 4; ++ch)
                st_shared_v4(base + wHh + (part >> 1) * 16384 + sw128(row, 4 * (part & 1) + ch),
                             pack_bf16(v[8 * ch], v[8 * ch + 1]), pack_bf16(v[8 * ch + 2], v[8 * ch + 3]),
                             pack_bf16(v[8 * ch + 4], v[8 * ch + 5]), pack_bf16(v[8 * ch + 6], v[8 * ch + 7]));
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tma_store_4d(&tmDQ, sm + wHh, 0, (int)(kv * GQ), (int)t0, (int)b);
            tma_store_4d(&tmDQ, sm + wHh + 16384, 64, (int)(kv * GQ), (int)t0, (int)b);
            bulk_commit();
        }
    }
    if (tid == 0) bulk_wait_all();  // the last dq tiles have left shared memory

    if (ok) {
        // dWf partial of the segment (lane = d, 16 feature columns per part) and dt partials
        float v[16];
        tmem_ld8(tb + lane_off + fDW + 16 * part, v);
        tmem_ld8(tb + lane_off + fDW + 16 * part + 8, v + 8);
        tmem_wait_ld();
        float* dst = dWp + ((size_t)seg * (size_t)U + (size_t)unit) * (size_t)(DH * 64) + row * 64 +
                     16 * part;
#pragma unroll
        for (int k = 0; k < 16; k += 4)
            *reinterpret_cast<float4*>(dst + k) =
                dw_init ? make_float4(v[k], v[k + 1], v[k + 2], v[k + 3])
                        : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        // dt partial: sum of a delta over the segment's rows of each head (head = row % 4),
        // in a fixed order: lanes of a warp, then the four lane quadrants
        if (part == 0) {
            float x = dts_acc;
            x += __shfl_xor_sync(0xffffffffu, x, 4);
            x += __shfl_xor_sync(0xffffffffu, x, 8);
            x += __shfl_xor_sync(0xffffffffu, x, 16);
            if (lane < 4) S.dts[quad][lane] = x;
        }
        __syncthreads();
        if (tid < GQ)
            dtp[((size_t)seg * (size_t)U + (size_t)unit) * GQ + tid] =
                (S.dts[0][tid] + S.dts[1][tid]) + (S.dts[2][tid] + S.dts[3][tid]);
    } else if (tid == 0) {
        if (mma_out) {
            mma_commit(&S.bar_fin);
            mbar_wait(&S.bar_fin, 0, kTimeout);
        }
        if (tma_out) mbar_wait(&S.bar_tma, ph_tma, kTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 512);
    }
}

// ---------------------------------------------------------------------------------------
// Reverse-direction walk of the backward on the tensor cores: the state parts of dk, dv of
// the delayed keys, the phi(k')-side of dB with its reverse cumulative sum inside the
// segment, and the dWf partial of the key side.  The segment is walked backwards in 32-token
// steps of 128 query rows (row = 4 token + head) and 32 delayed keys.  With the step's
// cumulative log-gates b (from its start), a reference rho = max(b_15, -60) per feature,
// a_i = e^{-lse_i}, delta_i = dy_i . y_i and the stored adjoint S (dH at the step start is
// e^{rho} (.) S):
//   S'   = e^{bl - rho + rho_next} (.) S_next             (the adjoint at the step end)
//   q^_i = phi(q_i) a_i e^{b_i - rho},   k^_t = phi(k'_t) e^{rho - b_t}
//   dphi(k')_t = e^{rho - b_t} (.) (S' v'_t + z' + sum_{i >= t} q^_i (dy_i . v'_t - delta_i))
//   dv'_t = S'^T k^_t + sum_{i >= t} (q^_i . k^_t) dy_i
//   S    = S' + q^^T dY,  z = z' - q^^T delta
// then dk' = du' Wf^T and dWf += k'^T du' from the feature-map backward du'.  The terms of
// dphi(k') that feed dB go in as high and low bf16 parts (dB feeds a nearly cancelling
// reverse cumulative sum); the decay factors stay in fp32.  Lanes hold features for the
// key-side accumulators ([f x keys]) and d for the outputs ([d x keys]).
constexpr uint32_t vR1 = 0, vR2 = 65536, vR3 = 98304, vK = 131072, vV = 139264, vW = 147456,
                   vG = 163840, vB = 172032, vPK = 188416, vDU = 204800, vX = 208896,
                   vSm = 221696;
struct VSmall {
    uint64_t bar_tma, bar_u, bar_g, bar_a, bar_v, bar_k, bar_fin;
    uint32_t tmem;
    volatile int abort;
    float z[128], rho_next[128], carry[128], rho[128], dlr[128], bl[128];
};
constexpr uint32_t kSmemRW = vSm + (uint32_t)sizeof(VSmall) + 1024;
static_assert(kSmemRW <= 232448, "shared memory budget");
// TMEM: S [0,128), G [128,160) (dphi(k') sums), C [160,192), A [192,224), dv'^T [224,256),
// dk'^T [256,288), dWf [288,352), U_q [352,416), U_k [416,480)
constexpr uint32_t vS = 0, vGc = 128, vC = 160, vA = 192, vDV = 224, vDK = 256, vDW = 288,
                   vUq = 352, vUk = 416;

// Byte offset of element (key t, row i) in a [32 keys x 128 rows] bf16 tile stored K-major
// over rows (two 64-row halves of 4 KB, 128-byte swizzle).
__device__ __forceinline__ uint32_t kt_off(int t, int i) {
    return (uint32_t)(i >> 6) * 4096u + sw128(t, (i & 63) >> 3) + (i & 7) * 2;
}

__device__ __forceinline__ bool fw_wait2(uint64_t* bar, uint32_t& ph, volatile int& abort,
                                         WsHeader* hdr, unsigned where) {
    bool fail = false;
    if (!mbar_try_wait(bar, ph)) {
        const long long t0 = clock64();
        while (!mbar_try_wait(bar, ph)) {
            if (abort || clock64() - t0 > kTimeout) {
                fail = true;
                break;
            }
        }
    }
    if (fail && !abort) {
        abort = 1;
        report(hdr, LIZARD_ERR_TIMEOUT, where);
    }
    if (!fail) ph ^= 1u;
    return !__syncthreads_or(fail);
}

// KEYF: the masked decay reading, as for the forward walk; the delayed keys' gate terms then
// go to a.kkey at the keys' own rows instead of into the reverse sum.
template <bool KEYF>
__global__ void __launch_bounds__(NT, 1)
    bwd_rwalk_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDY,
                 const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmG,
                 Plan p, BwdArgs a, const float* rows, const float* rev_rec, float* dB,
                 float* dWp, float* totp, const int* flags) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    VSmall& S = *reinterpret_cast<VSmall*>(sm + vSm);
    float* xa = reinterpret_cast<float*>(sm + vX);    // [4][128]
    float* xb = xa + 512;                             // [4][128]
    float* tn = xb + 512;                             // [32 keys][64 f]
    static_assert(vX + 4 * (512 + 512 + 2048 + 128) <= vSm, "exchange area");
    float* suk = reinterpret_cast<float*>(sm + vG);   // staged U_k rows [32][64]
    float* etab = reinterpret_cast<float*>(sm + vB);  // e^{b_t - rho} [32][128] fp32
    float* pk = reinterpret_cast<float*>(sm + vPK);   // phi(k') [32][128] fp32

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, part = warp >> 2;
    const int row = 32 * quad + lane;
    const int64_t unit = blockIdx.x, seg = blockIdx.y;
    const int64_t b = unit / p.Hkv, kv = unit % p.Hkv;
    const int64_t U = p.B * p.Hkv;
    const int64_t s0 = seg * p.seg_len, s1 = min64(p.L, s0 + p.seg_len);
    const int64_t c_first = s0 / CT, c_last = (s1 - 1) / CT;
    const int64_t nrow = p.B * p.L * p.Hq;
    WsHeader* hdr = (WsHeader*)a.ws;
    const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
    constexpr uint32_t kStepBytes = 2 * kTile + 8192u + 8192u + 8192u;  // q, dY, k', v', gates
    // a segment whose gates close too hard for the factored decays is the SIMT walk's
    if (flags[seg * U + unit] != 0) return;

    if (warp == 0) {
        tmem_alloc(&S.tmem, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&S.bar_tma, 1);
        mbar_init(&S.bar_u, 1);
        mbar_init(&S.bar_g, 1);
        mbar_init(&S.bar_a, 1);
        mbar_init(&S.bar_v, 1);
        mbar_init(&S.bar_k, 1);
        mbar_init(&S.bar_fin, 1);
        fence_mbar_init();
        S.abort = 0;
    }
    const bool last = seg == p.P - 1;
    const float* rec = last ? nullptr : rev_rec + ((size_t)seg * (size_t)U + (size_t)unit) * p.rec_floats;
    if (tid < 128) {
        S.z[tid] = rec ? rec[128 * DH + tid] : 0.0f;
        S.rho_next[tid] = 0.0f;
        S.carry[tid] = 0.0f;
    }
    if (rec) stage_record_in(sm + vR1, rec);  // vR1 is first written by the math threads
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = S.tmem;
    {
        float v[32];
        staged_row_read(sm + vR1, rec != nullptr, row, part, v);
        tmem_st32(tb + lane_off + vS + 32 * part, v);
        tmem_wait_st();
    }
    bool tma_out = false, mma_out = false;
    if (tid == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmDY);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmG);
        mbar_arrive_expect_tx(&S.bar_tma, kStepBytes + 16384u);
        tma_load_3d(sm + vW, &tmW, &S.bar_tma, 0, 0, (int)kv);
        load_delayed(sm + vK, &tmK, &S.bar_tma, kv, c_last, b);
        load_delayed(sm + vV, &tmV, &S.bar_tma, kv, c_last, b);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_4d(sm + vR2 + kb * 16384, &tmQ, &S.bar_tma, 64 * kb, (int)(kv * GQ),
                        (int)(c_last * CT), (int)b);
            tma_load_4d(sm + vR3 + kb * 16384, &tmDY, &S.bar_tma, 64 * kb, (int)(kv * GQ),
                        (int)(c_last * CT), (int)b);
        }
        tma_load_4d(sm + vG, &tmG, &S.bar_tma, 0, (int)kv, (int)(c_last * CT), (int)b);
        tma_out = true;
    }
    tc_fence_before();
    __syncthreads();
    const uint64_t dQk = kdesc(base + vR2), dDk = kdesc(base + vR3), dKk = kdesc(base + vK),
                   dVk = kdesc(base + vV), dWk = kdesc(base + vW);
    const uint64_t dWm = mndesc(base + vW, 16384), dDm = mndesc(base + vR3, 16384),
                   dKm = mndesc(base + vK, 4096);
    // R1 as the adjoint copy S' (K-major over d / MN-major over d), then as q^ (MN-major over f
    // for the f-row products, K-major over f for A = q^ k^^T)
    const uint64_t dS1h = kdesc(base + vR1), dS1l = kdesc(base + vR1 + 32768),
                   dS1hm = mndesc(base + vR1, 16384);
    const uint64_t dQhm = mndesc(base + vR1, 16384), dQlm = mndesc(base + vR1 + 32768, 16384),
                   dQhk = kdesc(base + vR1);
    // R2 after the query tile: k^ [32 keys][128 f] (8 KB), c high, c low, A^ (transposed tiles)
    const uint64_t dKh = kdesc(base + vR2), dCh = kdesc(base + vR2 + 8192),
                   dCl = kdesc(base + vR2 + 16384), dAh = kdesc(base + vR2 + 24576);
    const uint64_t dDUk = kdesc(base + vDU), dDUm = mndesc(base + vDU, 4096);
    uint32_t ph_tma = 0, ph_u = 0, ph_g = 0, ph_a = 0, ph_v = 0, ph_k = 0;
    bool ok = true, dw_init = false;

    for (int64_t c = c_last; c >= c_first; --c) {
        const int64_t t0 = c * CT;
        const int n = (int)min64(CT, s1 - t0);
        const bool more = c > c_first;
        if (KEYF && more && tid < 128) {  // the next step's key factors (32 rows), into L2
            const int64_t tn = t0 - CT + (tid >> 2);
            if (tn - WIN >= 0 && tn < s1)
                prefetch_l2(a.kdec + ((b * p.L + tn - WIN) * p.Hkv + kv) * 128 + 32 * (tid & 3));
        }
        ok = fw_wait2(&S.bar_tma, ph_tma, S.abort, hdr, 70);
        if (!ok) break;
        if (tid == 0) {
            tma_out = false;
            tc_fence_after();
            // (1) U_q, U_k of the delayed keys (rows 0..31), C = dY V_d^T
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t koff = ((j >> 2) * 16384 + (j & 3) * 32) >> 4;
                const uint32_t kdoff = ((j >> 2) * 4096 + (j & 3) * 32) >> 4;
                const uint64_t bw = dWm + ((j * 2048) >> 4);
                mma_bf16(tb + vUq, dQk + koff, bw, idesc_bf16(128, 64, false, true), j > 0);
                mma_bf16(tb + vUk, dKk + kdoff, bw, idesc_bf16(128, 64, false, true), j > 0);
                mma_bf16(tb + vC, dDk + koff, dVk + kdoff, idesc_bf16(128, 32, false, false), j > 0);
            }
            mma_commit(&S.bar_u);
            mma_out = true;
        }
        // (2) gates: b (fp32 table), rho = max(b_15, -60), decay of the stored adjoint
        const int gf = tid & 127, gq = tid >> 7;
        {
            const __nv_bfloat16* sg = (const __nv_bfloat16*)(sm + vG);
            float bt[8];
            float run = 0.0f;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const int tt = 8 * gq + t;
                run += tt < n ? log_sigmoid_f(__bfloat162float(sg[tt * 128 + gf])) : 0.0f;
                bt[t] = run;
            }
            xa[gq * 128 + gf] = run;
            __syncthreads();
            const float g0 = xa[gf], g1 = xa[128 + gf], g2 = xa[256 + gf], g3 = xa[384 + gf];
            const float off = gq == 0 ? 0.0f : gq == 1 ? g0 : gq == 2 ? g0 + g1 : (g0 + g1) + g2;
            // the decay factors of the step relative to rho, once per (token, feature): the
            // four heads of a token and both key-side phases read them from the table
            const float rh = fmaxf(g0 + g1, -60.0f);
#pragma unroll
            for (int t = 0; t < 8; ++t)
                etab[(8 * gq + t) * 128 + gf] = __expf(clamp80f(bt[t] + off - rh));
            if (gq == 0) {
                S.bl[gf] = ((g0 + g1) + g2) + g3;
                S.rho[gf] = rh;
            }
        }
        __syncthreads();
        // (3) S' = e^{bl - rho + rho_next} (.) S, as high and low bf16 parts for the
        //     key-side products; z' likewise
        {
            const int f = row;
            const float rh = S.rho[f];
            const float fac = __expf(S.bl[f] - rh + S.rho_next[f]);
            const int col = 32 * part;
            float v[32];
            tmem_ld32(tb + lane_off + vS + col, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] *= fac;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                const uint32_t off = (col / 64) * 16384 + sw128(f, (col & 63) / 8 + ch);
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) split2(v[8 * ch + 2 * e], v[8 * ch + 2 * e + 1], hi[e], lo[e]);
                st_shared_v4(base + vR1 + off, hi[0], hi[1], hi[2], hi[3]);
                st_shared_v4(base + vR1 + 32768 + off, lo[0], lo[1], lo[2], lo[3]);
            }
            tmem_st32(tb + lane_off + vS + col, v);
            tmem_wait_st();
            if (part == 0) S.z[f] *= fac;
        }
        ok = fw_wait2(&S.bar_u, ph_u, S.abort, hdr, 71);
        if (!ok) break;
        tc_fence_after();
        if (tid == 0) mma_out = false;
        if (quad == 0 && part < 2) {
            float w[32];
            tmem_ld32(tb + lane_off + vUk + 32 * part, w);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; k += 4)
                *reinterpret_cast<float4*>(suk + lane * 64 + 32 * part + k) =
                    make_float4(w[k], w[k + 1], w[k + 2], w[k + 3]);
        }
        // phi(q) of this thread's 16 u-values (features 16 part + k of both halves)
        float php[16], phn[16];
        {
            float u[16];
            tmem_ld8(tb + lane_off + vUq + 16 * part, u);
            tmem_ld8(tb + lane_off + vUq + 16 * part + 8, u + 8);
            tmem_wait_ld();
            float mx = -INFINITY, mn = -INFINITY;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                mx = fmaxf(mx, u[k]);
                mn = fmaxf(mn, -u[k]);
            }
            xa[part * 128 + row] = mx;
            xb[part * 128 + row] = mn;
            quad_sync(quad);
            mx = fmaxf(fmaxf(xa[row], xa[128 + row]), fmaxf(xa[256 + row], xa[384 + row]));
            mn = fmaxf(fmaxf(xb[row], xb[128 + row]), fmaxf(xb[256 + row], xb[384 + row]));
            float sp = 0.0f, sn = 0.0f;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                php[k] = __expf(u[k] - mx);
                phn[k] = __expf(-u[k] - mn);
                sp += php[k];
                sn += phn[k];
            }
            quad_sync(quad);
            xa[part * 128 + row] = sp;
            xb[part * 128 + row] = sn;
            quad_sync(quad);
            sp = (xa[row] + xa[128 + row]) + (xa[256 + row] + xa[384 + row]);
            sn = (xb[row] + xb[128 + row]) + (xb[256 + row] + xb[384 + row]);
            const float ip = 1.0f / sp, in = 1.0f / sn;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                php[k] *= ip;
                phn[k] *= in;
            }
        }
        __syncthreads();
        // (4) phi of the delayed keys (fp32, 16 threads per key) and k^ = phi e^{rho - b_t}
        //     (bf16, into R2: the query tile is consumed)
        {
            const int t = tid >> 4, sub = tid & 15;
            const bool dvalid = (t0 + t - WIN >= 0) && (t < n);
            float4 kd4[2] = {};  // the delayed key's own log factor (masked reading)
            if (KEYF && dvalid) {
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
                    kd4[kb] = *reinterpret_cast<const float4*>(
                        a.kdec + ((b * p.L + t0 + t - WIN) * p.Hkv + kv) * 128 + 64 * kb + 4 * sub);
            }
            const float4 u4 = *reinterpret_cast<const float4*>(suk + t * 64 + 4 * sub);
            const float u[4] = {u4.x, u4.y, u4.z, u4.w};
            float mx = fmaxf(fmaxf(u[0], u[1]), fmaxf(u[2], u[3]));
            float mn = fminf(fminf(u[0], u[1]), fminf(u[2], u[3]));
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) {
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            }
            float ep[4], en[4], sp = 0.0f, sn = 0.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                ep[e] = __expf(u[e] - mx);
                en[e] = __expf(mn - u[e]);
                sp += ep[e];
                sn += en[e];
            }
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) {
                sp += __shfl_xor_sync(0xffffffffu, sp, o);
                sn += __shfl_xor_sync(0xffffffffu, sn, o);
            }
            const float ip = dvalid ? 1.0f / sp : 0.0f, in = dvalid ? 1.0f / sn : 0.0f;
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
                const int f0 = 64 * kb + 4 * sub;
                float ph[4], kh[4], kf[4] = {1.0f, 1.0f, 1.0f, 1.0f};
                if (KEYF && dvalid) {
                    kf[0] = __expf(kd4[kb].x);
                    kf[1] = __expf(kd4[kb].y);
                    kf[2] = __expf(kd4[kb].z);
                    kf[3] = __expf(kd4[kb].w);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    ph[e] = kb == 0 ? ep[e] * ip : en[e] * in;
                    kh[e] = ph[e] * kf[e] * rcpf(etab[t * 128 + f0 + e]);  // e^{rho - b_t}
                }
                *reinterpret_cast<float4*>(pk + t * 128 + f0) = make_float4(ph[0], ph[1], ph[2], ph[3]);
                const uint32_t off = kb * 4096 + sw128(t, sub >> 1) + (sub & 1) * 8;
                asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(base + vR2 + off),
                             "r"(pack_bf16(kh[0], kh[1])), "r"(pack_bf16(kh[2], kh[3]))
                             : "memory");
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            // (5) G = S' V_d^T (high + low); dv'^T = S'^T k^^T
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t koff = ((j >> 2) * 16384 + (j & 3) * 32) >> 4;
                const uint32_t kdoff = ((j >> 2) * 4096 + (j & 3) * 32) >> 4;
                mma_bf16(tb + vGc, dS1h + koff, dVk + kdoff, idesc_bf16(128, 32, false, false), j > 0);
                mma_bf16(tb + vGc, dS1l + koff, dVk + kdoff, idesc_bf16(128, 32, false, false), 1);
                mma_bf16(tb + vDV, dS1hm + ((j * 2048) >> 4), dKh + kdoff,
                         idesc_bf16(128, 32, true, false), j > 0);
            }
            mma_commit(&S.bar_g);
            mma_out = true;
        }
        // (6) q^ = phi(q) a e^{b_i - rho} (high, low) into R1 once S' is read; c (high, low)
        const int ti = row >> 2;
        const int64_t ridx = (b * p.L + t0 + ti) * p.Hq + kv * GQ + (row & 3);
        const bool rv = ti < n;
        const float ar = rv ? rows[ridx] : 0.0f, dl = rv ? rows[nrow + ridx] : 0.0f;
        if (part == 0) S.dlr[row] = dl;  // delta per row for the z column sums
        ok = fw_wait2(&S.bar_g, ph_g, S.abort, hdr, 72);
        if (!ok) break;
        tc_fence_after();
        {
            const int fp = 16 * part, fn = 64 + 16 * part;
            uint32_t hp[8], lp[8], hn[8], ln[8];
#pragma unroll
            for (int k = 0; k < 16; k += 2) {
                float qp[2], qn[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int f1 = fp + k + h, f2 = fn + k + h;
                    qp[h] = php[k + h] * ar * etab[ti * 128 + f1];
                    qn[h] = phn[k + h] * ar * etab[ti * 128 + f2];
                }
                split2(qp[0], qp[1], hp[k / 2], lp[k / 2]);
                split2(qn[0], qn[1], hn[k / 2], ln[k / 2]);
            }
            // [f half][128 rows][64 f]: features fp.. are half 0, chunks 2 part, 2 part + 1
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const uint32_t o0 = h2 * 16384 + sw128(row, 2 * part),
                               o1 = h2 * 16384 + sw128(row, 2 * part + 1);
                const uint32_t* H = h2 == 0 ? hp : hn;
                const uint32_t* Lw = h2 == 0 ? lp : ln;
                st_shared_v4(base + vR1 + o0, H[0], H[1], H[2], H[3]);
                st_shared_v4(base + vR1 + o1, H[4], H[5], H[6], H[7]);
                st_shared_v4(base + vR1 + 32768 + o0, Lw[0], Lw[1], Lw[2], Lw[3]);
                st_shared_v4(base + vR1 + 32768 + o1, Lw[4], Lw[5], Lw[6], Lw[7]);
            }
            // c_it = dy_i . v'_t - delta_i for delayed keys t <= i, stored key-major
            float cv[8];
            tmem_ld8(tb + lane_off + vC + 8 * part, cv);
            tmem_wait_ld();
            __nv_bfloat16* ch = (__nv_bfloat16*)(sm + vR2 + 8192);
            __nv_bfloat16* cl = (__nv_bfloat16*)(sm + vR2 + 16384);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int t = 8 * part + e;
                const bool valid = rv && t <= ti && (t0 + t - WIN >= 0);
                const float x = valid ? cv[e] - dl : 0.0f;
                const __nv_bfloat16 xh = __float2bfloat16_rn(x);
                const uint32_t o = kt_off(t, row) / 2;
                ch[o] = xh;
                cl[o] = __float2bfloat16_rn(x - __bfloat162float(xh));
            }
        }
        // this step's dB rows (from the forward-direction walk) for phase (9), requested now so
        // the load overlaps the MMAs below
        float dbp[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int t = 8 * part + e;
            dbp[e] = t < n ? dB[((b * p.L + t0 + t) * p.Hkv + kv) * 128 + row] : 0.0f;
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            // (7) A = q^ k^^T; G += q^^T c (three parts); S += q^^T dY (two parts)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t koff = ((j >> 2) * 16384 + (j & 3) * 32) >> 4;
                const uint32_t kdoff = ((j >> 2) * 4096 + (j & 3) * 32) >> 4;
                mma_bf16(tb + vA, dQhk + koff, dKh + kdoff, idesc_bf16(128, 32, false, false), j > 0);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t ro = (j * 2048) >> 4;
                const uint32_t co = ((j >> 2) * 4096 + (j & 3) * 32) >> 4;
                mma_bf16(tb + vGc, dQhm + ro, dCh + co, idesc_bf16(128, 32, true, false), 1);
                mma_bf16(tb + vGc, dQhm + ro, dCl + co, idesc_bf16(128, 32, true, false), 1);
                mma_bf16(tb + vGc, dQlm + ro, dCh + co, idesc_bf16(128, 32, true, false), 1);
                mma_bf16(tb + vS, dQhm + ro, dDm + ro, idesc_bf16(128, 128, true, true), 1);
                mma_bf16(tb + vS, dQlm + ro, dDm + ro, idesc_bf16(128, 128, true, true), 1);
            }
            mma_commit(&S.bar_a);
        }
        // z <- z' - sum_rows q^ delta (from the bf16 parts the MMA reads)
        {
            const int f = tid & 127, gq2 = tid >> 7;
            const __nv_bfloat16* qh = (const __nv_bfloat16*)(sm + vR1);
            const __nv_bfloat16* ql = (const __nv_bfloat16*)(sm + vR1 + 32768);
            float zsum[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // four chains: the loads overlap
#pragma unroll
            for (int r = 32 * gq2; r < 32 * gq2 + 32; ++r) {
                const uint32_t o = ((f >> 6) * 16384 + sw128(r, (f & 63) >> 3) + (f & 7) * 2) / 2;
                zsum[r & 3] = fmaf(__bfloat162float(qh[o]) + __bfloat162float(ql[o]), S.dlr[r], zsum[r & 3]);
            }
            xa[gq2 * 128 + f] = (zsum[0] + zsum[1]) + (zsum[2] + zsum[3]);
        }
        ok = fw_wait2(&S.bar_a, ph_a, S.abort, hdr, 73);
        if (!ok) break;
        tc_fence_after();
        if (tid < 128) {
            const float zr = (xa[tid] + xa[128 + tid]) + (xa[256 + tid] + xa[384 + tid]);
            xb[tid] = S.z[tid];  // z' for dphi(k')
            S.z[tid] -= zr;
        }
        // (8) A^ (masked i >= t) key-major for dv' += dY^T A^
        {
            float av[8];
            tmem_ld8(tb + lane_off + vA + 8 * part, av);
            tmem_wait_ld();
            __nv_bfloat16* ah = (__nv_bfloat16*)(sm + vR2 + 24576);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int t = 8 * part + e;
                const bool valid = rv && t <= ti && (t0 + t - WIN >= 0);
                ah[kt_off(t, row) / 2] = __float2bfloat16_rn(valid ? av[e] : 0.0f);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < 8; ++j)
                mma_bf16(tb + vDV, dDm + ((j * 2048) >> 4),
                         dAh + ((((j >> 2) * 4096 + (j & 3) * 32)) >> 4),
                         idesc_bf16(128, 32, true, false), 1);
            mma_commit(&S.bar_v);
        }
        // (9) dphi(k') = e^{rho - b_t} (.) (G + z') for feature `row`, keys 8 part .. + 7;
        //     phi(k')-side of dB with the reverse cumulative sum; du'
        float dphi[8], phk[8];
        {
            const int f = row;
            float gv[8], kdl[8];
            if (KEYF) {  // the keys' log factors, every load issued before the first store
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int t = 8 * part + e;
                    const int64_t j = t0 + t - WIN;
                    kdl[e] = t < n && j >= 0 ? a.kdec[((b * p.L + j) * p.Hkv + kv) * 128 + f] : 0.0f;
                }
            }
            tmem_ld8(tb + lane_off + vGc + 8 * part, gv);
            tmem_wait_ld();
            const float zp = xb[f];
            float loc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int t = 8 * part + e;
                phk[e] = pk[t * 128 + f];
                dphi[e] = rcpf(etab[t * 128 + f]) * (gv[e] + zp);  // e^{rho - b_t} (G + z')
                if (KEYF) {
                    // masked reading: the key entered as c phi, so dphi = c (.) d(c phi); its
                    // gate term phi dphi belongs to the key's own row (kept apart in kkey)
                    const int64_t j = t0 + t - WIN;
                    if (t < n && j >= 0) {
                        const int64_t kidx = ((b * p.L + j) * p.Hkv + kv) * 128 + f;
                        dphi[e] *= __expf(kdl[e]);
                        a.kkey[kidx] = phk[e] * dphi[e];
                    }
                    loc[e] = t < n ? dbp[e] : 0.0f;
                } else {
                    loc[e] = t < n ? dbp[e] - phk[e] * dphi[e] : 0.0f;
                }
            }
            // suffix sums inside the part (keys descending), then across parts
            float suf[8];
            float run = 0.0f;
#pragma unroll
            for (int e = 7; e >= 0; --e) {
                run += loc[e];
                suf[e] = run;
            }
            xa[part * 128 + f] = run;  // part totals [4][128]
            __syncthreads();
            float cin = S.carry[f];
            for (int p2 = 3; p2 > part; --p2) cin += xa[p2 * 128 + f];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int t = 8 * part + e;
                if (t < n) dB[((b * p.L + t0 + t) * p.Hkv + kv) * 128 + f] = cin + suf[e];
            }
            __syncthreads();
            if (part == 0)
                S.carry[f] += (xa[f] + xa[128 + f]) + (xa[256 + f] + xa[384 + f]);
            // feature-map backward: per key, S_half = sum over the half of phi dphi
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float x = phk[e] * dphi[e];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                if (lane == 0) tn[2048 + quad * 32 + 8 * part + e] = x;  // [4 quads][32 keys]
            }
            __syncthreads();
        }
        {
            const int f = row;
            const int h = quad >> 1;  // 0: softmax(+u) half, 1: softmax(-u) half
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int t = 8 * part + e;
                const float Sh = tn[2048 + (2 * h) * 32 + t] + tn[2048 + (2 * h + 1) * 32 + t];
                const float term = phk[e] * (dphi[e] - Sh);
                if (h == 1) tn[t * 64 + (f - 64)] = term;
                else dphi[e] = term;  // quads 0, 1 keep the + term
            }
            __syncthreads();
            if (h == 0) {
                __nv_bfloat16* du = (__nv_bfloat16*)(sm + vDU);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int t = 8 * part + e;
                    const float v = dphi[e] - tn[t * 64 + f];
                    du[(sw128(t, f >> 3) + (f & 7) * 2) / 2] = __float2bfloat16_rn(v);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            // (10) dk'^T = Wf du'^T; dWf += k'^T du'
#pragma unroll
            for (int j = 0; j < 4; ++j)
                mma_bf16(tb + vDK, dWk + ((j * 32) >> 4), dDUk + ((j * 32) >> 4),
                         idesc_bf16(128, 32, false, false), j > 0);
#pragma unroll
            for (int j = 0; j < 2; ++j)
                mma_bf16(tb + vDW, dKm + ((j * 2048) >> 4), dDUm + ((j * 2048) >> 4),
                         idesc_bf16(128, 64, true, true), (dw_init || j > 0) ? 1u : 0u);
            mma_commit(&S.bar_k);
        }
        dw_init = true;
        ok = fw_wait2(&S.bar_v, ph_v, S.abort, hdr, 74);
        if (!ok) break;
        ok = fw_wait2(&S.bar_k, ph_k, S.abort, hdr, 75);
        if (!ok) break;
        tc_fence_after();
        if (tid == 0) {
            mma_out = false;
            if (more) {
                // every tile of this step is consumed: the previous step's copies start
                mbar_arrive_expect_tx(&S.bar_tma, kStepBytes);
                load_delayed(sm + vK, &tmK, &S.bar_tma, kv, c - 1, b);
                load_delayed(sm + vV, &tmV, &S.bar_tma, kv, c - 1, b);
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
                    tma_load_4d(sm + vR2 + kb * 16384, &tmQ, &S.bar_tma, 64 * kb, (int)(kv * GQ),
                                (int)((c - 1) * CT), (int)b);
                    tma_load_4d(sm + vR3 + kb * 16384, &tmDY, &S.bar_tma, 64 * kb, (int)(kv * GQ),
                                (int)((c - 1) * CT), (int)b);
                }
                tma_load_4d(sm + vG, &tmG, &S.bar_tma, 0, (int)kv, (int)((c - 1) * CT), (int)b);
                tma_out = true;
            }
        }
        // (11) dk, dv of the delayed keys (lane = d, keys 8 part .. + 7)
        {
            float kv8[8], vv8[8];
            tmem_ld8(tb + lane_off + vDK + 8 * part, kv8);
            tmem_ld8(tb + lane_off + vDV + 8 * part, vv8);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int t = 8 * part + e;
                const int64_t j = t0 + t - WIN;
                if (t < n && j >= 0) {
                    const int64_t o = ((b * p.L + j) * p.Hkv + kv) * DH + row;
                    ((__nv_bfloat16*)a.dk)[o] = __float2bfloat16_rn(kv8[e]);
                    ((__nv_bfloat16*)a.dv)[o] = __float2bfloat16_rn(vv8[e]);
                }
            }
        }
        if (tid < 128) S.rho_next[tid] = S.rho[tid];
        tc_fence_before();
        __syncthreads();
    }

    if (ok) {
        float v[16];
        tmem_ld8(tb + lane_off + vDW + 16 * part, v);
        tmem_ld8(tb + lane_off + vDW + 16 * part + 8, v + 8);
        tmem_wait_ld();
        float* dst = dWp + ((size_t)(p.Pmax + seg) * (size_t)U + (size_t)unit) * (size_t)(DH * 64) +
                     row * 64 + 16 * part;
#pragma unroll
        for (int k = 0; k < 16; k += 4)
            *reinterpret_cast<float4*>(dst + k) =
                dw_init ? make_float4(v[k], v[k + 1], v[k + 2], v[k + 3])
                        : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (tid < 128) totp[((size_t)seg * (size_t)U + (size_t)unit) * 128 + tid] = S.carry[tid];
    } else if (tid == 0) {
        if (mma_out) {
            mma_commit(&S.bar_fin);
            mbar_wait(&S.bar_fin, 0, kTimeout);
        }
        if (tma_out) mbar_wait(&S.bar_tma, ph_tma, kTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 512);
    }
}

}  // namespace

bool bwd_win_tc_supported(const Plan& p) {
    return p.dtype == LIZARD_BF16 && p.d == DH && p.G == GQ && p.w == WIN &&
           p.L < ((int64_t)1 << 30) && p.B * p.Hkv <= 65535 && tc::encode_fn() != nullptr;
}

cudaError_t launch_bwd_fwalk_tc(const Plan& p, const BwdArgs& a, float* wsf, size_t o_rows,
                                size_t o_fwd, size_t o_dB, size_t o_dW, size_t o_dt,
                                const int* flags, cudaStream_t s) {
    alignas(64) CUtensorMap mq, md, mk, mv, mw, mg, mdq;
    const cuuint64_t B = (cuuint64_t)p.B, L = (cuuint64_t)p.L, Hq = (cuuint64_t)p.Hq,
                     Hkv = (cuuint64_t)p.Hkv;
    {
        const cuuint64_t dims[4] = {DH, Hq, L, B};
        const cuuint64_t str[3] = {DH * 2, Hq * DH * 2, L * Hq * DH * 2};
        const cuuint32_t box[4] = {64, GQ, CT, 1};
        if (!tc::make_map(&mq, a.q, 4, dims, str, box)) return cudaErrorInvalidValue;
        if (!tc::make_map(&md, a.dy, 4, dims, str, box)) return cudaErrorInvalidValue;
        if (!tc::make_map(&mdq, a.dq, 4, dims, str, box)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[4] = {DH, Hkv, L, B};
        const cuuint64_t str[3] = {DH * 2, Hkv * DH * 2, L * Hkv * DH * 2};
        const cuuint32_t box[4] = {64, 1, CT, 1};
        if (!tc::make_map(&mk, a.k, 4, dims, str, box)) return cudaErrorInvalidValue;
        if (!tc::make_map(&mv, a.v, 4, dims, str, box)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[4] = {128, Hkv, L, B};
        const cuuint64_t str[3] = {128 * 2, Hkv * 128 * 2, L * Hkv * 128 * 2};
        const cuuint32_t box[4] = {128, 1, CT, 1};
        if (!tc::make_map(&mg, a.g, 4, dims, str, box, false)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {64, DH, Hkv};
        const cuuint64_t str[2] = {64 * 2, DH * 64 * 2};
        const cuuint32_t box[3] = {64, DH, 1};
        if (!tc::make_map(&mw, a.Wf, 3, dims, str, box)) return cudaErrorInvalidValue;
    }
    auto walk = a.kdec != nullptr ? bwd_fwalk_tc<true> : bwd_fwalk_tc<false>;
    cudaError_t e = cudaFuncSetAttribute(walk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemFW);
    if (e != cudaSuccess) return e;
    walk<<<dim3((unsigned)(p.B * p.Hkv), (unsigned)p.P), NT, kSmemFW, s>>>(
        mq, md, mk, mv, mw, mg, mdq, p, a, wsf + o_rows, wsf + o_fwd, wsf + o_dB, wsf + o_dW,
        wsf + o_dt, flags);
    return cudaGetLastError();
}

cudaError_t launch_bwd_rwalk_tc(const Plan& p, const BwdArgs& a, float* wsf, size_t o_rows,
                                size_t o_rev, size_t o_dB, size_t o_dW, size_t o_tot,
                                const int* flags, cudaStream_t s) {
    alignas(64) CUtensorMap mq, md, mk, mv, mw, mg;
    const cuuint64_t B = (cuuint64_t)p.B, L = (cuuint64_t)p.L, Hq = (cuuint64_t)p.Hq,
                     Hkv = (cuuint64_t)p.Hkv;
    {
        const cuuint64_t dims[4] = {DH, Hq, L, B};
        const cuuint64_t str[3] = {DH * 2, Hq * DH * 2, L * Hq * DH * 2};
        const cuuint32_t box[4] = {64, GQ, CT, 1};
        if (!tc::make_map(&mq, a.q, 4, dims, str, box)) return cudaErrorInvalidValue;
        if (!tc::make_map(&md, a.dy, 4, dims, str, box)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[4] = {DH, Hkv, L, B};
        const cuuint64_t str[3] = {DH * 2, Hkv * DH * 2, L * Hkv * DH * 2};
        const cuuint32_t box[4] = {64, 1, CT, 1};
        if (!tc::make_map(&mk, a.k, 4, dims, str, box)) return cudaErrorInvalidValue;
        if (!tc::make_map(&mv, a.v, 4, dims, str, box)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[4] = {128, Hkv, L, B};
        const cuuint64_t str[3] = {128 * 2, Hkv * 128 * 2, L * Hkv * 128 * 2};
        const cuuint32_t box[4] = {128, 1, CT, 1};
        if (!tc::make_map(&mg, a.g, 4, dims, str, box, false)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {64, DH, Hkv};
        const cuuint64_t str[2] = {64 * 2, DH * 64 * 2};
        const cuuint32_t box[3] = {64, DH, 1};
        if (!tc::make_map(&mw, a.Wf, 3, dims, str, box)) return cudaErrorInvalidValue;
    }
    auto walk = a.kdec != nullptr ? bwd_rwalk_tc<true> : bwd_rwalk_tc<false>;
    cudaError_t e = cudaFuncSetAttribute(walk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemRW);
    if (e != cudaSuccess) return e;
    walk<<<dim3((unsigned)(p.B * p.Hkv), (unsigned)p.P), NT, kSmemRW, s>>>(
        mq, md, mk, mv, mw, mg, p, a, wsf + o_rows, wsf + o_rev, wsf + o_dB, wsf + o_dW,
        wsf + o_tot, flags);
    return cudaGetLastError();
}

bool bwd_rev_local_tc_supported(const Plan& p) {
    return bwd_win_tc_supported(p) && p.D == 128;
}

cudaError_t launch_bwd_rev_local_tc(const Plan& p, const BwdArgs& a, const float* rows,
                                    float* rev_rec, cudaStream_t s) {
    if (p.P <= 1) return cudaSuccess;
    alignas(64) CUtensorMap mq, md, mw, mg;
    const cuuint64_t B = (cuuint64_t)p.B, L = (cuuint64_t)p.L, Hq = (cuuint64_t)p.Hq,
                     Hkv = (cuuint64_t)p.Hkv;
    {
        const cuuint64_t dims[4] = {DH, Hq, L, B};
        const cuuint64_t str[3] = {DH * 2, Hq * DH * 2, L * Hq * DH * 2};
        const cuuint32_t box[4] = {64, GQ, CT, 1};
        if (!tc::make_map(&mq, a.q, 4, dims, str, box)) return cudaErrorInvalidValue;
        if (!tc::make_map(&md, a.dy, 4, dims, str, box)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[4] = {128, Hkv, L, B};
        const cuuint64_t str[3] = {128 * 2, Hkv * 128 * 2, L * Hkv * 128 * 2};
        const cuuint32_t box[4] = {128, 1, CT, 1};
        if (!tc::make_map(&mg, a.g, 4, dims, str, box, false)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {64, DH, Hkv};
        const cuuint64_t str[2] = {64 * 2, DH * 64 * 2};
        const cuuint32_t box[3] = {64, DH, 1};
        if (!tc::make_map(&mw, a.Wf, 3, dims, str, box)) return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(bwd_rev_local_tc,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemRev);
    if (e != cudaSuccess) return e;
    bwd_rev_local_tc<<<dim3((unsigned)(p.B * p.Hkv), (unsigned)(p.P - 1)), NT, kSmemRev, s>>>(
        mq, md, mw, mg, p, a, rows, rev_rec);
    return cudaGetLastError();
}

cudaError_t launch_bwd_win_tc(const Plan& p, const BwdArgs& a, const float* rows, bool keys,
                              cudaStream_t s) {
    alignas(64) CUtensorMap mq, md, mk, mv;
    const cuuint64_t B = (cuuint64_t)p.B, L = (cuuint64_t)p.L, Hq = (cuuint64_t)p.Hq,
                     Hkv = (cuuint64_t)p.Hkv;
    {
        const cuuint64_t dims[4] = {DH, Hq, L, B};
        const cuuint64_t str[3] = {DH * 2, Hq * DH * 2, L * Hq * DH * 2};
        const cuuint32_t box[4] = {64, GQ, CT, 1};
        if (!tc::make_map(&mq, a.q, 4, dims, str, box)) return cudaErrorInvalidValue;
        if (!tc::make_map(&md, a.dy, 4, dims, str, box)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[4] = {DH, Hkv, L, B};
        const cuuint64_t str[3] = {DH * 2, Hkv * DH * 2, L * Hkv * DH * 2};
        const cuuint32_t box[4] = {64, 1, keys ? 128u : (cuuint32_t)KR, 1};
        if (!tc::make_map(&mk, a.k, 4, dims, str, box)) return cudaErrorInvalidValue;
        if (!tc::make_map(&mv, a.v, 4, dims, str, box)) return cudaErrorInvalidValue;
    }
    const dim3 grid((unsigned)((p.L + 127) / 128), (unsigned)(p.B * p.Hkv));
    cudaError_t e;
    if (keys) {
        e = cudaFuncSetAttribute(bwd_win_kv_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemKV);
        if (e != cudaSuccess) return e;
        bwd_win_kv_tc<<<grid, NT, kSmemKV, s>>>(mq, md, mk, mv, p, a, rows);
    } else {
        e = cudaFuncSetAttribute(bwd_win_q_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemQ);
        if (e != cudaSuccess) return e;
        bwd_win_q_tc<<<grid, NT, kSmemQ, s>>>(mq, md, mk, mv, p, a, rows);
    }
    return cudaGetLastError();
}

}  // namespace lz
