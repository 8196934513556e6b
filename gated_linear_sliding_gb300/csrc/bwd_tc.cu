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

// Bounded wait by every thread; all return the same verdict.
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

    for (int n = 0; ok && n < nq; ++n) {
        const int buf = n & 1;
        const int64_t c = c_first + n, q0 = c * CT;
        // rows of this tile: lse and delta (columns of S^T)
        if (tid < 128) {
            const int64_t i = q0 + (tid >> 2);
            const int64_t idx = (b * p.L + i) * p.Hq + kv * GQ + (tid & 3);
            slse[buf * 128 + tid] = i < p.L ? a.lse[idx] * kLog2e : 0.0f;
            sdel[buf * 128 + tid] = i < p.L ? rows[nrow + idx] : 0.0f;
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

    for (int n = 0; ok && n < nq; ++n) {
        const int64_t c = c0 + n, q0 = c * CT;
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
        const float ls = rv ? a.lse[idx] * kLog2e : 0.0f;
        const float dl = rv ? rows[nrow + idx] : 0.0f;
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
        if (rv) add_store_row((__nv_bfloat16*)a.dq + idx * DH + 32 * part, v, true);
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

}  // namespace

bool bwd_win_tc_supported(const Plan& p) {
    return p.dtype == LIZARD_BF16 && p.d == DH && p.G == GQ && p.w == WIN &&
           p.L < ((int64_t)1 << 30) && p.B * p.Hkv <= 65535 && tc::encode_fn() != nullptr;
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
