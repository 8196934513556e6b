// Tensor-core forward of the Lizard token mixer on sm_103a: tcgen05 MMAs with TMEM
// accumulators, operands staged by TMA in 128-byte-swizzled shared memory.
//
// Covers the LLaMA-3-8B / Mistral-7B-shaped layers: bf16, d = D = 128, four query
// heads per KV head, window w = 64.  Other shapes take the SIMT path.
//
// Lizard summary (gist.science/ko/paper/2507.09025):
//   sec. 2-A-1  gated linear attention, state S_i = Gamma_i (.) S_{i-1} + phi(k) v^T
//               (here the key that leaves the window enters the state);
//   sec. 2-A-2  sliding-window softmax with meta-memory scalars in the denominator;
//   sec. 2-C    the Hedgehog map is non-negative, so the gate products move to log
//               space and fold into the query and key sides, which turns the chunk
//               into plain low-precision GEMMs on the tensor cores.
//
// One CTA per (batch, KV head, segment); it walks its segment 32 tokens at a time.  Sixteen
// math warps do the softmaxes, masks and decay tables; one control warp issues every TMA
// copy and MMA and hands results over through mbarriers, so the next step's projections run
// while the math warps finish the current step.
// The 128 query rows of a step are (token, head) pairs, row = 4 * token + head, so
// the four heads of a group share every key-side operand.  Per step:
//   b_t   = sum_{s<=t} log sigmoid(g_s)  (fp32, chunk-local), reference r = b_15
//   q~_i  = phi(q_i) e^{b_i - r} e^{-m_i}          m_i = row shift (window, sinks)
//   k~_t  = phi(k_{t-w}) e^{r - b_t}                (delayed key of stream step t)
//   O_i   = q~_i (e^{r} (.) H) + P_win V_ring + [q~ k~^T (.) causal] V_delayed
//   H    <- e^{b_31} (.) H + (phi(k_{t-w}) e^{b_31 - b_t})^T V_delayed
//   y_i   = O_i / (sum P_win + sum P_intra + q~_i.(e^{r} z) + sum_m e^{t_m - m_i})
// Every gate factor is e^{difference of cumulative log-gates}, formed as a running product of
// Gamma = sigmoid(g) or 1/Gamma = 1 + e^{-g} over the tokens in between; relative to the
// step midpoint r each factor stays within the decay of one 16-token half.  That factored form
// is exact only while no half decays too far (a factor e^{b_i - r} of a half that decays by
// e^-200 does not exist in fp32).  A step on which some 8-token quarter of some feature
// decays by more than e^-36 therefore leaves this kernel: the CTA writes the state it would
// start that step from into its own record slot, marks the slot with the step, and stops; the
// exact SIMT tail walk (fwd_simt_tail) finishes the segment from there.  On the steps this
// kernel does run, every factor lies in [e^-72, e^72].
//
// TMEM columns: H [0,128)  scores S [128,256) (intra scores A reuse [128,160))
//               U_q [256,320)  U_k [320,384) (then P_win, bf16 pairs)  O [384,512).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"
#include "tc_util.cuh"

namespace lz {
namespace {

using namespace sm100;
using namespace tc;

constexpr int NW = 16;        // math warps: warp w owns TMEM lanes 32(w%4).., w/4 picks a 32-column part
constexpr int NS = 32 * NW;   // math threads
constexpr int NT = NS + 32;   // plus one control warp that issues every TMA copy and MMA
constexpr int CT = 32;        // tokens per step
constexpr int GQ = 4;         // query heads per KV head
constexpr int DH = 128;       // head dim
constexpr int DF = 128;       // phi dim
constexpr int WIN = 64;       // window
constexpr int MMAX = 64;      // sinks per head

// shared-memory map (bytes from a 1024-aligned base); later uses of a region in a step follow
// the arrow
constexpr uint32_t oQ = 0;         // q tile, K-major [128 rows][128 d]
constexpr uint32_t oQt = 32768;    // q~, K-major [128][128] -> y tile for the TMA store
constexpr uint32_t oK = 65536;     // key ring: 4 slots x 32 keys, K-major over d
constexpr uint32_t oV = 98304;     // value ring: same bytes, read MN-major (N = d)
constexpr uint32_t oW = 131072;    // Wf [128 d rows][64 features], MN-major B
constexpr uint32_t oHs = 147456;   // e^{r} (.) H in bf16, [128 feature rows][128 d], MN-major B
constexpr uint32_t oKi = 180224;   // k~ (intra), K-major [32 keys][128] -> P_intra sums [4][128]
constexpr uint32_t oKu = 188416;   // row exchange (max, u-extreme, u-sum) [3][4][128] -> k~ (update)
constexpr uint32_t oE = 196608;    // Eq, Ek tables (bf16 [32][128] each) -> P_intra
constexpr uint32_t oG = 212992;    // gate logits [32][128] bf16 -> staged U_k rows [32][64] fp32
constexpr uint32_t oSmall = 221184;

struct Small {
    uint64_t bar_tma;  // copies landed
    uint64_t bar_u;    // U_k (U_q, window scores) in TMEM
    uint64_t bar_q;    // q~, k~ in shared memory (math warps -> control)
    uint64_t bar_a;    // intra scores in TMEM
    uint64_t bar_p;    // P_intra in shared memory (math warps -> control)
    uint64_t bar_o;    // outputs and state update done
    uint64_t bar_fin;  // drain after an abort
    uint32_t tmem;
    volatile int abort;
    float z[DF], zs[DF], cf[DF];
    float gpart[4][DF];            // per-quarter products of Gamma (later: z partial sums)
    float gipart[4][DF];           // per-quarter products of 1/Gamma
    float ps[4][128], pg[4][128];  // per-part window and state denominators of each row
    float tmax[GQ];                // max(t_m) log2(e) per head (at least the minimum shift)
    float sexp[GQ];                // sum_m 2^{t_m log2(e) - tmax} per head
};
constexpr uint32_t kSmemBytes = oSmall + (uint32_t)sizeof(Small) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

// TMEM column bases: H [0,128), window scores S [128,256) (the intra scores A reuse its first
// 32 columns once S is read), U_q [256,320), U_k [320,384), O [384,512).  Once the delayed
// keys' U_k rows are staged, the window probabilities P_win (128 rows x 128 keys, bf16 pairs)
// take U_k's columns and feed the output MMA from TMEM.  O has columns of its own so the next
// step's projections can run while the epilogue still reads O.
constexpr uint32_t cH = 0, cS = 128, cA = 128, cUq = 256, cUk = 320, cPw = 320, cO = 384;

// Largest product of 1/Gamma over an 8-token quarter of a step this kernel runs (e^36): the
// midpoint factors of its steps then stay within [e^-72, e^72].
constexpr float kQuarterMax = 4.311231547115195e15f;
// Lower bound of the row shift m in this kernel: q~ = phi(q) e^{-m} e^{b_i - r} / sum stays
// below e^{8} e^{72}, inside the bf16 range.
constexpr float kTcMinShift = -8.0f;

// Decay tables [32 tokens][128 features] bf16: the 16-byte chunks of token t's row are
// XOR-swizzled by t, so rows read by neighbouring tokens fall in different banks.
__device__ __forceinline__ int eidx(int t, int f) { return t * DF + (((f >> 3) ^ (t & 7)) << 3) + (f & 7); }


// Barrier among the 128 math threads (4 warps) that share one TMEM lane quadrant.
__device__ __forceinline__ void quad_sync(int quad) {
    asm volatile("bar.sync %0, 128;" ::"r"(1 + quad) : "memory");
}
// Barrier among the math threads (the control warp never joins it).
__device__ __forceinline__ void math_sync() { asm volatile("bar.sync 5, 512;" ::: "memory"); }
// Barrier among the math threads that also returns whether any of them passed `pred`.
__device__ __forceinline__ bool math_any(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 6, 512, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}

// Bounded wait for a barrier phase that also gives up as soon as another thread aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Small& S) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (S.abort) return false;
        if (clock64() - t0 > kTimeout) return false;
    }
    return true;
}

// Math threads: every one of them calls this; all return the same verdict.
__device__ __forceinline__ bool math_wait(uint64_t* bar, uint32_t& ph, Small& S, WsHeader* hdr,
                                          unsigned where) {
    const bool fail = !wait_or_abort(bar, ph, S);
    if (fail && !S.abort) {
        S.abort = 1;
        report(hdr, LIZARD_ERR_TIMEOUT, where);
    }
    ph ^= 1u;
    return !math_any(fail);
}

// Control thread.
__device__ __forceinline__ bool ctl_wait(uint64_t* bar, uint32_t& ph, Small& S, WsHeader* hdr,
                                         unsigned where) {
    if (!wait_or_abort(bar, ph, S)) {
        if (!S.abort) {
            S.abort = 1;
            report(hdr, LIZARD_ERR_TIMEOUT, where);
        }
        return false;
    }
    ph ^= 1u;
    return true;
}

// Bytes one step's copies bring: key and value slots, the gate tile (and the query tile).
constexpr uint32_t kStepBytes = 16384u + 8192u + 32768u;

// Key/value slot of chunk c (and its query tile), on a barrier phase that expects `expect`
// bytes in all (the gate tile follows separately).
// Token coordinates are tok0 + 32 c: tok0 is the first row of a packed sequence (its maps span
// every row, batch coordinate bco = 0) or 0 in a dense batch (bco = b).
__device__ __forceinline__ void issue_kvq_loads(uint8_t* sm, uint64_t* bar, const CUtensorMap* tmQ,
                                                const CUtensorMap* tmK, const CUtensorMap* tmV,
                                                int64_t c, int64_t kv, int64_t tok0, int64_t b,
                                                uint32_t expect) {
    const int slot = (int)(c & 3);
    const int t0 = (int)(tok0 + c * 32);
    sm100::mbar_arrive_expect_tx(bar, expect);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
        sm100::tma_load_4d(sm + oK + kb * 16384 + slot * 4096, tmK, bar, 64 * kb, (int)kv, t0, (int)b);
        sm100::tma_load_4d(sm + oV + kb * 16384 + slot * 4096, tmV, bar, 64 * kb, (int)kv, t0, (int)b);
        sm100::tma_load_4d(sm + oQ + kb * 16384, tmQ, bar, 64 * kb, (int)(kv * 4), t0, (int)b);
    }
}

__device__ __forceinline__ void issue_gate_load(uint8_t* sm, uint64_t* bar, const CUtensorMap* tmG,
                                                int64_t c, int64_t kv, int64_t tok0, int64_t b) {
    sm100::tma_load_4d(sm + oG, tmG, bar, 0, (int)kv, (int)(tok0 + c * 32), (int)b);
}

// The control warp: lane 0 issues the copies and the three MMA groups of every step and
// hands each result to the math warps through an mbarrier.  The next step's query tile and
// ring slot are loaded as soon as this step's projections have read theirs, its gate tile
// once the delayed keys' feature map has consumed the staged U_k rows.
__device__ __forceinline__ void control_loop(uint8_t* sm, uint32_t base, uint32_t tb, Small& S,
                                             WsHeader* hdr, const CUtensorMap* tmQ,
                                             const CUtensorMap* tmK, const CUtensorMap* tmV,
                                             const CUtensorMap* tmW, const CUtensorMap* tmG,
                                             int64_t c_begin, int64_t c_end, int64_t kv,
                                             int64_t tok0, int64_t b) {
    const uint64_t dQ = kdesc(base + oQ), dQt = kdesc(base + oQt), dK = kdesc(base + oK),
                   dKi = kdesc(base + oKi), dE = kdesc(base + oE);
    const uint64_t dW = mndesc(base + oW, 16384), dHs = mndesc(base + oHs, 16384),
                   dV = mndesc(base + oV, 16384), dKu = mndesc(base + oKu, 4096);
    uint32_t ph_tma = 0, ph_u = 0, ph_q = 0, ph_p = 0, ph_o = 0;
    bool tma_out = false, mma_out = false;
    int64_t gate_due = -1;  // chunk whose gate tile its barrier phase still waits for
    if (c_begin < c_end) {
        // the first step's operands, Wf and the two chunks before the segment, all on one
        // phase; chunks before the sequence start are not loaded (their ring slots keep the
        // zeros written at entry)
        const int64_t c_prev = c_begin - 2 > 0 ? c_begin - 2 : 0;
        issue_kvq_loads(sm, &S.bar_tma, tmQ, tmK, tmV, c_begin, kv, tok0, b,
                        kStepBytes + 16384u + (uint32_t)(c_begin - c_prev) * 16384u);
        issue_gate_load(sm, &S.bar_tma, tmG, c_begin, kv, tok0, b);
        tma_load_3d(sm + oW, tmW, &S.bar_tma, 0, 0, (int)kv);
        for (int64_t cc = c_prev; cc < c_begin; ++cc) {
            const int slot = (int)(cc & 3);
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
                tma_load_4d(sm + oK + kb * 16384 + slot * 4096, tmK, &S.bar_tma, 64 * kb, (int)kv,
                            (int)(tok0 + cc * CT), (int)b);
                tma_load_4d(sm + oV + kb * 16384 + slot * 4096, tmV, &S.bar_tma, 64 * kb, (int)kv,
                            (int)(tok0 + cc * CT), (int)b);
            }
        }
        tma_out = true;
    }
    for (int64_t c = c_begin; c < c_end; ++c) {
        const int slot_d = (int)((c - 2) & 3);
        const int slot_x = (int)((c + 1) & 3);  // three steps old: no key of the window
        const bool more = c + 1 < c_end;
        if (!ctl_wait(&S.bar_tma, ph_tma, S, hdr, 2)) break;
        tma_out = false;
        tc_fence_after();
        // feature-map projections (and window scores) of this step
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t koff = ((j >> 2) * 16384 + (j & 3) * 32) >> 4;
            const uint64_t bw = dW + ((j * 2048) >> 4);
            mma_bf16(tb + cUk, dK + koff, bw, idesc_bf16(128, 64, false, true), j > 0);
            mma_bf16(tb + cUq, dQ + koff, bw, idesc_bf16(128, 64, false, true), j > 0);
            mma_bf16(tb + cS, dQ + koff, dK + koff, idesc_bf16(128, 128, false, false), j > 0);
        }
        mma_commit(&S.bar_u);
        mma_out = true;
        if (!ctl_wait(&S.bar_u, ph_u, S, hdr, 9)) break;
        // the query tile and the ring slot of chunk c-3 are free: next step's copies start
        if (more) {
            issue_kvq_loads(sm, &S.bar_tma, tmQ, tmK, tmV, c + 1, kv, tok0, b, kStepBytes);
            tma_out = true;
            gate_due = c + 1;
        }
        if (!ctl_wait(&S.bar_q, ph_q, S, hdr, 6)) break;
        tc_fence_after();
        if (more) {
            issue_gate_load(sm, &S.bar_tma, tmG, c + 1, kv, tok0, b);
            gate_due = -1;
        }
        const uint64_t dVd = dV + ((slot_d * 4096) >> 4);
        // intra-step scores A = q~ k~^T
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t qoff = ((j >> 2) * 16384 + (j & 3) * 32) >> 4;
            const uint32_t koff = ((j >> 2) * 4096 + (j & 3) * 32) >> 4;
            mma_bf16(tb + cA, dQt + qoff, dKi + koff, idesc_bf16(128, 32, false, false), j > 0);
        }
        mma_commit(&S.bar_a);
        // the parts of O that do not wait for P_intra: q~ H_s + P_win V_ring, and the state
        // update H += k~u^T V_delayed, run while the math warps mask A
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t aoff = ((j >> 2) * 16384 + (j & 3) * 32) >> 4;
            mma_bf16(tb + cO, dQt + aoff, dHs + ((j * 2048) >> 4), idesc_bf16(128, 128, false, true),
                     j > 0);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if ((j >> 1) == slot_x) continue;  // P_win is zero there; the slot is reloading
            mma_bf16_ts(tb + cO, tb + cPw + 8 * j, dV + ((j * 2048) >> 4),
                        idesc_bf16(128, 128, false, true), 1);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j)
            mma_bf16(tb + cH, dKu + ((j * 2048) >> 4), dVd + ((j * 2048) >> 4),
                     idesc_bf16(128, 128, true, true), 1);
        if (!ctl_wait(&S.bar_p, ph_p, S, hdr, 7)) break;
        tc_fence_after();
        // O += P_intra V_delayed
#pragma unroll
        for (int j = 0; j < 2; ++j)
            mma_bf16(tb + cO, dE + ((j * 32) >> 4), dVd + ((j * 2048) >> 4),
                     idesc_bf16(128, 128, false, true), 1);
        mma_commit(&S.bar_o);
        if (!ctl_wait(&S.bar_o, ph_o, S, hdr, 8)) break;
        mma_out = false;
    }
    if (S.abort) {
        // let copies and MMAs still in flight land before the CTA exits
        if (mma_out) {
            mma_commit(&S.bar_fin);
            mbar_wait(&S.bar_fin, 0, kTimeout);
        }
        if (tma_out) {
            if (gate_due >= 0) issue_gate_load(sm, &S.bar_tma, tmG, gate_due, kv, tok0, b);
            mbar_wait(&S.bar_tma, ph_tma, kTimeout);
        }
    }
}

// KEYF: the masked decay reading (each entering key's factor e^{kd} folded into its decay
// table); a separate instantiation, so the other readings' code is not touched by it.
template <bool KEYF>
__global__ void __launch_bounds__(NT, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmW,
                  const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmY,
                  Plan p, FwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    Small& S = *reinterpret_cast<Small*>(sm + oSmall);
    float* xpm = reinterpret_cast<float*>(sm + oKu);         // [4][128] window partial max
    float* xum = xpm + 512;                                   // [4][128] u partial extreme
    float* xus = xpm + 1024;                                  // [4][128] u partial sum
    float* spi = reinterpret_cast<float*>(sm + oKi);         // [4][128] P_intra partial sums
    float* suk = reinterpret_cast<float*>(sm + oG);          // [32][64] staged U_k rows

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, part = (warp >> 2) & 3;
    const int row = 32 * quad + lane;
    const int64_t unit = blockIdx.x, seg = blockIdx.y;
    const int64_t b = unit / p.Hkv, kv = unit % p.Hkv;
    const int64_t U = p.B * p.Hkv;
    // sequence b: rows row0 .. row0 + len - 1; TMA coordinates (tok0 + t, bco)
    const int64_t row0 = seq_row0(p, b), len = seq_len(p, b);
    const int64_t tok0 = p.cu != nullptr ? row0 : 0, bco = p.cu != nullptr ? 0 : b;
    const int64_t s0 = seg * p.seg_len;
    const int64_t s1 = min64(len, s0 + p.seg_len);
    WsHeader* hdr = (WsHeader*)a.header;
    const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
    const int64_t c_begin = s0 / CT, c_end = (s1 + CT - 1) / CT;
    if (s0 >= len) {
        // a segment past the end of a shorter packed sequence: nothing to walk; its record
        // slot tells the tail walk so (after the scan, which writes the same slots)
        grid_dep_launch();
        grid_dep_wait();
        if (tid == 0)
            a.seg[((size_t)(seg * p.rec_step) * (size_t)U + (size_t)unit) * p.rec_floats + DF * DH +
                  DF] = __int_as_float(-1);
        return;
    }

    if (warp == 0) {
        tmem_alloc(&S.tmem, 512);
        tmem_relinquish();
    }
    grid_dep_launch();  // the tail walk may be launched now (it waits for this grid's end)
    if (tid == 0) {
        mbar_init(&S.bar_tma, 1);
        mbar_init(&S.bar_u, 1);
        mbar_init(&S.bar_q, 1);
        mbar_init(&S.bar_a, 1);
        mbar_init(&S.bar_p, 1);
        mbar_init(&S.bar_o, 1);
        mbar_init(&S.bar_fin, 1);
        fence_mbar_init();
        S.abort = 0;
    }
    if (warp == NW && lane == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmG);
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmY);
    }
    if (tid < GQ) {
        const float* t = a.sinks + (kv * GQ + tid) * p.M;
        float tm = kTcMinShift;
        for (int mm = 0; mm < p.M; ++mm) tm = fmaxf(tm, t[mm]);
        float se = 0.0f;
        for (int mm = 0; mm < p.M; ++mm) se += ex2f((t[mm] - tm) * kLog2e);
        S.tmax[tid] = tm * kLog2e;
        S.sexp[tid] = se;
    }
    // The starting state passes through shared memory (the rings' bytes, zeroed afterwards):
    // coalesced 16-byte loads, and each row's 16-byte chunks XOR-swizzled by the row so the
    // per-row reads below are free of bank conflicts.
    const float* rec =
        seg > 0 ? a.seg + ((size_t)(seg * p.rec_step) * (size_t)U + (size_t)unit) * p.rec_floats
                : nullptr;
    grid_dep_wait();  // the records come from the scan launched just before
    if (rec != nullptr) stage_record_in(sm + oK, rec);
    if (tid < DF) S.z[tid] = rec ? rec[DF * DH + tid] : 0.0f;
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = S.tmem;
    if (warp < NW) {
        // starting state H into TMEM (fp32 master copy), lane = feature f, column = d
        float v[32];
        staged_row_read(sm + oK, rec != nullptr, row, part, v);
        tmem_st32(tb + lane_off + cH + 32 * part, v);
        tmem_wait_st();
    }
    __syncthreads();
    // zero both rings: P_win is 0 on masked keys, but 0 times non-finite stale bits is NaN
    for (int e = tid; e < 65536 / 16; e += NT) st_shared_v4(base + oK + e * 16, 0u, 0u, 0u, 0u);
    fence_async_smem();
    __syncthreads();

    if (warp == NW) {
        if (lane == 0)
            control_loop(sm, base, tb, S, hdr, &tmQ, &tmK, &tmV, &tmW, &tmG, c_begin, c_end,
                               kv, tok0, bco);
        __syncwarp();
    } else {
        uint32_t ph_tma = 0, ph_u = 0, ph_a = 0, ph_o = 0;
        bool ok = true;
        int64_t stop = -1;  // the step handed to the exact tail walk, if any

        for (int64_t c = c_begin; c < c_end; ++c) {
            const int64_t t0 = c * CT;
            const int n = (int)min64(CT, s1 - t0);
            const int slot_d = (int)((c - 2) & 3);

            const int gf = tid & (DF - 1), gq = tid >> 7;  // phase (2): feature, quarter
            // masked decay reading: the delayed key of each of the thread's tokens enters with
            // its phi scaled by the product of the w gates it saw in the window, e^{kd}, folded
            // into its decay factor in phase (2).  Loaded before the wait for the step's tiles,
            // and the next step's factors are fetched into L2 meanwhile.
            float kl[CT / 4];  // log factors (0 for a token with no key entering)
#pragma unroll
            for (int t = 0; t < CT / 4; ++t) {
                const int64_t j = t0 + (CT / 4) * gq + t - WIN;
                kl[t] = KEYF && j >= 0 && (CT / 4) * gq + t < n
                            ? a.kdec[((row0 + j) * p.Hkv + kv) * DF + gf]
                            : 0.0f;
            }
            if (KEYF) {
#pragma unroll
                for (int t = 0; t < CT / 4; ++t) {
                    const int64_t j = t0 + CT + (CT / 4) * gq + t - WIN;
                    if (j >= 0 && j + WIN < s1)
                        prefetch_l2(a.kdec + ((row0 + j) * p.Hkv + kv) * DF + gf);
                }
            }

            // (1) this step's keys, values, gates (and queries) have landed; the control warp
            //     has started the feature-map projections and window scores
            ok = math_wait(&S.bar_tma, ph_tma, S, hdr, 2);
            if (!ok) break;

            // (2) gates: four threads per feature, one per 8-token quarter.  Every decay factor
            //     of the step relative to r = b_15 is a running product of Gamma = sigmoid(g) or
            //     of 1/Gamma = 1 + e^{-g} over the tokens between (no logarithm)
            float ig[CT / 4];  // 1/Gamma of the thread's tokens (Gamma itself is rcp of it)
            float pig = 1.0f;
            {
                const __nv_bfloat16* sg = (const __nv_bfloat16*)(sm + oG);
#pragma unroll
                for (int t = 0; t < CT / 4; ++t) {
                    const int tt = (CT / 4) * gq + t;
                    const float x = __bfloat162float(sg[tt * DF + gf]);
                    ig[t] = tt < n ? 1.0f + ex2f(-x * kLog2e) : 1.0f;  // past the end: Gamma = 1
                    pig *= ig[t];
                }
                S.gpart[gq][gf] = rcpf(pig);
                S.gipart[gq][gf] = pig;
            }
            // a quarter that decays by more than e^-36 (or a non-finite product) on any feature:
            // the step goes to the exact tail walk, before anything of it is written
            if (math_any(!(pig <= kQuarterMax))) {
                stop = c;
                if (tid == 0) S.abort = 2;  // releases the control warp without an error
                break;
            }
            {
                __nv_bfloat16* Eq = (__nv_bfloat16*)(sm + oE);
                __nv_bfloat16* Ek = (__nv_bfloat16*)(sm + oE + 8192);
                if (gq < 2) {
                    // t < 16: Eq = prod_{s=t+1..15} 1/Gamma_s, Ek = prod_{s=t+1..15} Gamma_s
                    float sq = gq == 0 ? S.gipart[1][gf] : 1.0f, sk = gq == 0 ? S.gpart[1][gf] : 1.0f;
#pragma unroll
                    for (int t = CT / 4 - 1; t >= 0; --t) {
                        const int tt = (CT / 4) * gq + t;
                        Eq[eidx(tt, gf)] = __float2bfloat16_rn(sq);
                        Ek[eidx(tt, gf)] = __float2bfloat16_rn(KEYF ? sk * __expf(kl[t]) : sk);
                        sq *= ig[t];
                        sk *= rcpf(ig[t]);
                    }
                } else {
                    // t >= 16: Eq = prod_{s=16..t} Gamma_s, Ek = prod_{s=16..t} 1/Gamma_s
                    float pq = gq == 3 ? S.gpart[2][gf] : 1.0f, pk = gq == 3 ? S.gipart[2][gf] : 1.0f;
#pragma unroll
                    for (int t = 0; t < CT / 4; ++t) {
                        const int tt = (CT / 4) * gq + t;
                        pq *= rcpf(ig[t]);
                        pk *= ig[t];
                        Eq[eidx(tt, gf)] = __float2bfloat16_rn(pq);
                        Ek[eidx(tt, gf)] = __float2bfloat16_rn(KEYF ? pk * __expf(kl[t]) : pk);
                    }
                }
                if (gq == 0) {
                    const float g0 = S.gpart[0][gf], g1 = S.gpart[1][gf];
                    S.cf[gf] = S.gpart[2][gf] * S.gpart[3][gf];  // e^{b_31 - r}
                    S.zs[gf] = (g0 * g1) * S.z[gf];               // e^{r} z
                }
            }

            // (3) the state's bf16 copy scaled by e^{r} for the readout, and the fp32 master
            //     decayed by e^{b_31} (TMEM columns no MMA in flight touches)
            {
                const int f = row;
                const float er = S.gpart[0][f] * S.gpart[1][f];
                const float el = er * (S.gpart[2][f] * S.gpart[3][f]);
                const int col = 32 * part;
                float v[32];
                tmem_ld32(tb + lane_off + cH + col, v);
                tmem_wait_ld();
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    const int nchunk = (col & 63) / 8 + ch;
                    st_shared_v4(base + oHs + (col / 64) * 16384 + sw128(f, nchunk),
                                 pack_bf16(er * v[8 * ch], er * v[8 * ch + 1]),
                                 pack_bf16(er * v[8 * ch + 2], er * v[8 * ch + 3]),
                                 pack_bf16(er * v[8 * ch + 4], er * v[8 * ch + 5]),
                                 pack_bf16(er * v[8 * ch + 6], er * v[8 * ch + 7]));
                }
#pragma unroll
                for (int k = 0; k < 32; ++k) v[k] *= el;
                tmem_st32(tb + lane_off + cH + col, v);
                tmem_wait_st();
            }
            // the previous step's y tile has left the q~ buffer before anyone writes q~ again
            // (the barrier of the wait below orders this before the q~ writes of phase (4))
            if (tid == 0) bulk_wait_read();
            ok = math_wait(&S.bar_u, ph_u, S, hdr, 3);
            if (!ok) break;
            tc_fence_after();

            // (4) window softmax over the ring slot `part`, the query feature map, U_k staging.
            //     Exponents are kept in base 2: m2 = m log2(e).
            const int i = row >> 2, hh = row & 3;
            const int64_t qa = t0 + i;
            const bool qv = i < n;
            float m2 = 0.0f;
            if (quad == slot_d && part < 2) {
                float w[32];
                tmem_ld32(tb + lane_off + cUk + 32 * part, w);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 32; k += 4)
                    *reinterpret_cast<float4*>(suk + lane * 64 + 32 * part + k) =
                        make_float4(w[k], w[k + 1], w[k + 2], w[k + 3]);
            }
            {
                // keys of ring slot `part` are tokens 32 (c - age) + u; the slot that is three
                // steps old, and slots before the sequence start, hold no key of the window
                const int age = (int)((c - part) & 3);
                const bool live = age <= 2 && c >= age;  // same for the whole warp
                const int sib = part ^ 1;
                const float s2 = p.scale * kLog2e;
                uint32_t vm = 0;  // bit u: key u of the slot is in this row's window
                if (live && qv) {
                    const int64_t kbase = (c - age) * CT;
                    const int64_t lo = max64(0, qa - WIN + 1 - kbase);
                    const int64_t hi = min64(31, qa - kbase);
                    if (hi >= lo) vm = (uint32_t)(((2ull << hi) - 1ull) & ~((1ull << lo) - 1ull));
                }
                // first pass: row maxima (scores and u); the rows are read again from TMEM
                // after the exchange rather than held in registers across it
                {
                    float pmax = -INFINITY;
                    if (live) {
                        float sv[32];
                        tmem_ld32(tb + lane_off + cS + 32 * part, sv);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            pmax = fmaxf(pmax, ((vm >> k) & 1u) ? sv[k] * s2 : -INFINITY);
                    }
                    float uv[32];
                    tmem_ld32(tb + lane_off + cUq + 32 * (part & 1), uv);
                    tmem_wait_ld();
                    // parts 0, 1 take softmax(+u) over features [0, 64), parts 2, 3 softmax(-u)
                    float uext = -INFINITY;
                    if (part < 2) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) uext = fmaxf(uext, uv[k]);
                    } else {
#pragma unroll
                        for (int k = 0; k < 32; ++k) uext = fmaxf(uext, -uv[k]);
                    }
                    xpm[part * 128 + row] = pmax;
                    xum[part * 128 + row] = uext;
                }
                // the exchanges below stay within the 4 warps of a lane quadrant (one row per
                // lane); the staged U_k rows are read after the barrier at the end of this phase
                tc_fence_before();
                quad_sync(quad);
                m2 = fmaxf(fmaxf(fmaxf(xpm[row], xpm[128 + row]), fmaxf(xpm[256 + row], xpm[384 + row])),
                           S.tmax[hh]);
                float psum = 0.0f;
                tc_fence_after();  // the staged U_k reads of this quad precede the P_win writes
                uint32_t pw[16];
                if (live) {
                    float sv[32];
                    tmem_ld32(tb + lane_off + cS + 32 * part, sv);
                    tmem_wait_ld();
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        float pv[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int k = 8 * ch + e;
                            pv[e] = ex2f(((vm >> k) & 1u) ? fmaf(sv[k], s2, -m2) : -INFINITY);
                        }
                        pw[4 * ch] = round_pair(pv[0], pv[1]);
                        pw[4 * ch + 1] = round_pair(pv[2], pv[3]);
                        pw[4 * ch + 2] = round_pair(pv[4], pv[5]);
                        pw[4 * ch + 3] = round_pair(pv[6], pv[7]);
                        psum += ((pv[0] + pv[1]) + (pv[2] + pv[3])) + ((pv[4] + pv[5]) + (pv[6] + pv[7]));
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) pw[e] = 0u;
                }
                // keys 32 part + u of this row -> P_win columns 16 part + u / 2
                tmem_st16(tb + lane_off + cPw + 16 * part, pw);
                S.ps[part][row] = psum;
                const float f2 = part < 2 ? kLog2e : -kLog2e;
                const float cst = -fmaxf(xum[part * 128 + row], xum[sib * 128 + row]) * kLog2e;
                float uv[32];
                tmem_ld32(tb + lane_off + cUq + 32 * (part & 1), uv);
                tmem_wait_ld();
                float usum = 0.0f;
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    uv[k] = ex2f(fmaf(uv[k], f2, cst));
                    usum += uv[k];
                }
                xus[part * 128 + row] = usum;
                quad_sync(quad);
                // q~ = phi(q) e^{b_i - r} e^{-m}: features [32 part, 32 part + 32)
                const float sc = ex2f(-m2) / (xus[part * 128 + row] + xus[sib * 128 + row]);
                float pg = 0.0f;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    const int f0 = 32 * part + 8 * ch;
                    uint32_t w0, w1, w2, w3;
                    ld_shared_v4(base + oE + (uint32_t)eidx(i, f0) * 2u, w0, w1, w2, w3);
                    float eq[8], qv8[8];
                    unpack8(w0, w1, w2, w3, eq);
                    const float4 za = *reinterpret_cast<const float4*>(&S.zs[f0]);
                    const float4 zb = *reinterpret_cast<const float4*>(&S.zs[f0 + 4]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) qv8[e] = uv[8 * ch + e] * sc * eq[e];
                    const uint32_t q0 = round_pair(qv8[0], qv8[1]), q1 = round_pair(qv8[2], qv8[3]),
                                   q2 = round_pair(qv8[4], qv8[5]), q3 = round_pair(qv8[6], qv8[7]);
                    pg = fmaf(qv8[0], za.x, pg);
                    pg = fmaf(qv8[1], za.y, pg);
                    pg = fmaf(qv8[2], za.z, pg);
                    pg = fmaf(qv8[3], za.w, pg);
                    pg = fmaf(qv8[4], zb.x, pg);
                    pg = fmaf(qv8[5], zb.y, pg);
                    pg = fmaf(qv8[6], zb.z, pg);
                    pg = fmaf(qv8[7], zb.w, pg);
                    st_shared_v4(base + oQt + (part >> 1) * 16384 + sw128(row, 4 * (part & 1) + ch),
                                 q0, q1, q2, q3);
                }
                S.pg[part][row] = pg;
                tmem_wait_st();
            }
            math_sync();

            // (5) phi of the delayed keys (the ring slot two steps back) from the staged U_k
            //     rows: 16 threads per key, 4 u-values each -> k~ for the intra scores and the
            //     update
            {
                const int t = tid >> 4, sub = tid & 15;
                const bool dvalid = (t0 + t - WIN >= 0) && (t < n);
                const float4 u4 = *reinterpret_cast<const float4*>(suk + t * 64 + 4 * sub);
                const float u[4] = {u4.x, u4.y, u4.z, u4.w};
                float mx = fmaxf(fmaxf(u[0], u[1]), fmaxf(u[2], u[3]));
                float mn = fminf(fminf(u[0], u[1]), fminf(u[2], u[3]));
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) {
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
                }
                const float cmx = -mx * kLog2e, cmn = mn * kLog2e;
                float ep[4], en[4], sp = 0.0f, sn = 0.0f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    ep[e] = ex2f(fmaf(u[e], kLog2e, cmx));
                    en[e] = ex2f(fmaf(u[e], -kLog2e, cmn));
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
                    const int f0 = 64 * kb + 4 * sub;  // features f0..f0+3 (kb 0: softmax(u), 1: -u)
                    // the four decay factors are 8 contiguous bytes of the swizzled table
                    const uint2 e2 = *reinterpret_cast<const uint2*>(sm + oE + 8192 + eidx(t, f0) * 2);
                    const float ek[4] = {__uint_as_float(e2.x << 16), __uint_as_float(e2.x & 0xffff0000u),
                                         __uint_as_float(e2.y << 16), __uint_as_float(e2.y & 0xffff0000u)};
                    const float4 cf4 = *reinterpret_cast<const float4*>(&S.cf[f0]);
                    const float cf[4] = {cf4.x, cf4.y, cf4.z, cf4.w};
                    float ki[4], ku[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float ph = kb == 0 ? ep[e] * ip : en[e] * in;
                        ki[e] = ph * ek[e];
                        ku[e] = ki[e] * cf[e];
                    }
                    const uint32_t off = kb * 4096 + sw128(t, sub >> 1) + (sub & 1) * 8;
                    {
                        const uint32_t a0 = pack_bf16(ki[0], ki[1]), a1 = pack_bf16(ki[2], ki[3]);
                        asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(base + oKi + off),
                                     "r"(a0), "r"(a1)
                                     : "memory");
                    }
                    const uint32_t b0 = pack_bf16(ku[0], ku[1]), b1 = pack_bf16(ku[2], ku[3]);
                    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(base + oKu + off), "r"(b0),
                                 "r"(b1)
                                 : "memory");
                }
            }
            fence_async_smem();
            tc_fence_before();
            math_sync();
            if (tid == 0) mbar_arrive(&S.bar_q);

            // z <- e^{b_31} z + sum_t k~u_t (read back from the bf16 tile the MMA uses): four
            // threads per feature sum 8 tokens each into the quarter slots phase (3) has read
            {
                const int f = tid & (DF - 1), zq = tid >> 7;
                float zsum = 0.0f;
                const __nv_bfloat16* ku = (const __nv_bfloat16*)(sm + oKu);
#pragma unroll
                for (int t = 8 * zq; t < 8 * zq + 8; ++t) {
                    const uint32_t off = (f >> 6) * 4096 + sw128(t, (f & 63) >> 3) + (f & 7) * 2;
                    zsum += __bfloat162float(ku[off / 2]);
                }
                S.gpart[zq][f] = zsum;
            }
            // the parts of this row's shared normaliser known before P_intra: window, state
            // and sink terms (while the intra-score MMA runs)
            const float den0 = (S.ps[0][row] + S.ps[1][row]) + (S.ps[2][row] + S.ps[3][row]) +
                               (S.pg[0][row] + S.pg[1][row]) + (S.pg[2][row] + S.pg[3][row]) +
                               ex2f(S.tmax[hh] - m2) * S.sexp[hh];  // sum_m e^{t_m - m}
            float inv = 0.0f;
            {
                ok = math_wait(&S.bar_a, ph_a, S, hdr, 4);
                if (!ok) break;
                tc_fence_after();
                if (tid < DF)  // e^{b_31} z = e^{b_31 - r} e^{r} z
                    S.z[tid] = fmaf(S.cf[tid], S.zs[tid],
                                    (S.gpart[0][tid] + S.gpart[1][tid]) + (S.gpart[2][tid] + S.gpart[3][tid]));
                // (6) P_intra: columns t in [8 part, 8 part + 8)
                float av[8];
                tmem_ld8(tb + lane_off + cA + 8 * part, av);
                tmem_wait_ld();
                float pv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int t = 8 * part + e;
                    const bool valid = qv && t <= i && (t0 + t - WIN >= 0);
                    pv[e] = valid ? av[e] : 0.0f;
                }
                const uint32_t w0 = round_pair(pv[0], pv[1]), w1 = round_pair(pv[2], pv[3]),
                               w2 = round_pair(pv[4], pv[5]), w3 = round_pair(pv[6], pv[7]);
                st_shared_v4(base + oE + sw128(row, part), w0, w1, w2, w3);
                spi[part * 128 + row] =
                    ((pv[0] + pv[1]) + (pv[2] + pv[3])) + ((pv[4] + pv[5]) + (pv[6] + pv[7]));
                fence_async_smem();
                tc_fence_before();
                math_sync();
                if (tid == 0) mbar_arrive(&S.bar_p);
                // the shared normaliser of this row, while the output MMAs run
                if (qv) {
                    const float den = den0 + ((spi[row] + spi[128 + row]) + (spi[256 + row] + spi[384 + row]));
                    inv = 1.0f / den;
                    if (part == 0 && a.lse != nullptr)
                        a.lse[(row0 + qa) * p.Hq + kv * GQ + hh] = m2 * kLn2 + __logf(den);
                }
            }
            ok = math_wait(&S.bar_o, ph_o, S, hdr, 5);
            if (!ok) break;
            tc_fence_after();

            // (7) epilogue: y = O / den over columns [32 part, 32 part + 32) into the y tile
            //     (q~'s buffer, free once the output MMAs are done), then one TMA store.  The
            //     last, partial step of a packed sequence stores its valid rows directly: the
            //     tile's other rows are the next sequence's.
            {
                float ov[32];
                const int col = 32 * part;
                tmem_ld32(tb + lane_off + cO + col, ov);
                tmem_wait_ld();
                const bool direct = p.cu != nullptr && n < CT;
                uint4* yrow = reinterpret_cast<uint4*>(
                    (__nv_bfloat16*)a.y + ((row0 + qa) * p.Hq + kv * GQ + hh) * DH + col);
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    const uint32_t w0 = pack_bf16(ov[8 * ch] * inv, ov[8 * ch + 1] * inv),
                                   w1 = pack_bf16(ov[8 * ch + 2] * inv, ov[8 * ch + 3] * inv),
                                   w2 = pack_bf16(ov[8 * ch + 4] * inv, ov[8 * ch + 5] * inv),
                                   w3 = pack_bf16(ov[8 * ch + 6] * inv, ov[8 * ch + 7] * inv);
                    if (!direct)
                        st_shared_v4(base + oQt + (part >> 1) * 16384 + sw128(row, 4 * (part & 1) + ch),
                                     w0, w1, w2, w3);
                    else if (qv)
                        yrow[ch] = make_uint4(w0, w1, w2, w3);
                }
                fence_async_smem();
                math_sync();
                if (tid == 0 && !direct) {
                    // rows past the end of a dense batch's sequence fall outside the tensor
                    tma_store_4d(&tmY, sm + oQt, 0, (int)(kv * GQ), (int)(tok0 + t0), (int)bco);
                    tma_store_4d(&tmY, sm + oQt + 16384, 64, (int)(kv * GQ), (int)(tok0 + t0),
                                 (int)bco);
                    bulk_commit();
                }
            }
        }
        if (tid == 0) bulk_wait_all();

        // Record slot of this CTA (the one it read its starting state from, or slot 0): the
        // state handed to the tail walk, and in the first log-decay word the step it starts at
        // (-1: nothing to finish).  Written on every call, so no earlier call's mark survives.
        float* ho = a.seg + ((size_t)(seg * p.rec_step) * (size_t)U + (size_t)unit) * p.rec_floats;
        if (ok && stop >= 0) {
            float v[32];
            const int col = 32 * part;
            tmem_ld32(tb + lane_off + cH + col, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; k += 4)
                *reinterpret_cast<float4*>(ho + row * DH + col + k) =
                    make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
            if (tid < DF) ho[DF * DH + tid] = S.z[tid];
        }
        if (tid == 0) ho[DF * DH + DF] = __int_as_float(ok && stop >= 0 ? (int)stop : -1);

        if (ok && stop < 0 && a.S_out != nullptr && s1 == len) {
            // final state of the last segment: the decode hand-off
            float* dstH = a.S_out + unit * DF * DH;
            float* dstz = a.z_out + unit * DF;
            {
                float v[32];
                const int col = 32 * part;
                tmem_ld32(tb + lane_off + cH + col, v);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 32; k += 4)
                    *reinterpret_cast<float4*>(dstH + row * DH + col + k) =
                        make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
                if (tid < DF) dstz[tid] = S.z[tid];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 512);
    }
}

// ---------------------------------------------------------------------------------------
// Segment pass: the state a segment leaves behind when it starts from zero,
//   H_seg = sum_t e^{b_end - b_t} (.) phi(k_{t-w}) v_{t-w}^T,   z_seg likewise,
// (b = cumulative log-sigmoid gate from the segment start) and its total log-decay, for
// every segment but the last.  Steps of 128 tokens: the delayed keys of a step fill one
// 128-row MMA tile, so U_k = k Wf and the update H += k~^T v are one MMA group each, and the
// state is decayed once per 128 tokens.
constexpr int LT = 128;  // tokens per segment-pass step
constexpr uint32_t lK = 0;         // delayed keys [2 halves][128 rows][64 d], K-major
constexpr uint32_t lV = 32768;     // delayed values, same layout, read MN-major
constexpr uint32_t lG = 65536;     // gate logits [128 tokens][128 features] bf16
constexpr uint32_t lW = 98304;     // Wf, MN-major B
constexpr uint32_t lKu = 114688;   // k~ = phi(k) e^{b_end - b_t}, [2 halves][128 tokens][64 f]
constexpr uint32_t lE = 147456;    // e^{b_end - b_t} fp32 [128 tokens][EKR] (padded rows)
constexpr int EKR = DF + 4;        // row pitch (floats) of lE: rows land in distinct bank groups
constexpr uint32_t lKul = lE;      // low bf16 part of k~ (layout of lKu), over lE once it is read
constexpr uint32_t lX = lE + 128 * EKR * 4;  // exchanges: u-extreme, u-sum, gate and z quarters
constexpr uint32_t lSmall = lX + 8192;

struct LSmall {
    uint64_t bar_k, bar_v, bar_g, bar_u, bar_h, bar_fin;
    uint32_t tmem;
    volatile int abort;
    float z[DF], el[DF];
};
static_assert(lKul % 1024 == 0 && 32768 <= 128 * EKR * 4, "segment-pass layout");
constexpr uint32_t kLocalSmem = lSmall + sizeof(LSmall) + 1024;
static_assert(kLocalSmem <= 232448, "shared memory budget");
constexpr int NL = 512;  // threads of the segment pass

// Bounded wait by every thread of the segment pass; all return the same verdict.
__device__ __forceinline__ bool local_wait(uint64_t* bar, uint32_t& ph, LSmall& S, WsHeader* hdr,
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

// Token t of a 128-row tile: absolute row coordinate t (tok0 added by the caller), batch b.
__device__ __forceinline__ void local_load(uint8_t* dst, const CUtensorMap* tm, uint64_t* bar,
                                           int64_t kv, int64_t t, int64_t b) {
    mbar_arrive_expect_tx(bar, 32768u);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb)
        tma_load_4d(dst + kb * 16384, tm, bar, 64 * kb, (int)kv, (int)t, (int)b);
}

template <bool KEYF>
__global__ void __launch_bounds__(NL, 1)
    fwd_tc_local(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmG,
                 Plan p, FwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    LSmall& S = *reinterpret_cast<LSmall*>(sm + lSmall);
    float* xum = reinterpret_cast<float*>(sm + lX);  // [4][128] u extreme per (part, key)
    float* xus = xum + 512;                          // [4][128] u sums
    float* gpart = xum + 1024;                       // [4][128] gate quarter sums
    float* zq = xum + 1536;                          // [4][128] z quarter sums

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, part = warp >> 2;
    const int row = 32 * quad + lane;
    const int64_t unit = blockIdx.x, seg = blockIdx.y;
    const int64_t b = unit / p.Hkv, kv = unit % p.Hkv;
    const int64_t U = p.B * p.Hkv;
    const int64_t row0 = seq_row0(p, b), len = seq_len(p, b);
    const int64_t tok0 = p.cu != nullptr ? row0 : 0, bco = p.cu != nullptr ? 0 : b;
    const int64_t s0 = seg * p.seg_len;
    const int64_t s1 = min64(len, s0 + p.seg_len);
    // (a segment past the end of a shorter packed sequence walks nothing: zero record)
    const int64_t nsteps = s1 > s0 ? (s1 - s0 + LT - 1) / LT : 0;
    // the first tile's delayed keys and values before a packed sequence's start are the
    // previous sequence's rows: zeroed in shared memory (a dense batch reads zero fill there)
    const bool zero_pre = p.cu != nullptr && s0 < WIN;
    WsHeader* hdr = (WsHeader*)a.header;
    const uint32_t lane_off = (uint32_t)(32 * quad) << 16;

    if (warp == 0) {
        tmem_alloc(&S.tmem, 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&S.bar_k, 1);
        mbar_init(&S.bar_v, 1);
        mbar_init(&S.bar_g, 1);
        mbar_init(&S.bar_u, 1);
        mbar_init(&S.bar_h, 1);
        mbar_init(&S.bar_fin, 1);
        fence_mbar_init();
        S.abort = 0;
    }
    if (tid < DF) S.z[tid] = 0.0f;
    grid_dep_launch();  // the scan may be launched now (it waits for this grid's end)
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = S.tmem;
    const uint32_t cHl = 0, cUl = 128;  // TMEM: H [0,128), U_k [128,192)
    const uint64_t dK = kdesc(base + lK);
    const uint64_t dW = mndesc(base + lW, 16384), dV = mndesc(base + lV, 16384),
                   dKu = mndesc(base + lKu, 16384), dKul = mndesc(base + lKul, 16384);
    {
        float v[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = 0.0f;
        tmem_st32(tb + lane_off + cHl + 32 * part, v);
        tmem_wait_st();
    }
    bool k_out = false, v_out = false, g_out = false, mma_out = false;
    if (tid == 0 && nsteps > 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmG);
        mbar_arrive_expect_tx(&S.bar_k, 32768u + 16384u);
        tma_load_3d(sm + lW, &tmW, &S.bar_k, 0, 0, (int)kv);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
            tma_load_4d(sm + lK + kb * 16384, &tmK, &S.bar_k, 64 * kb, (int)kv,
                        (int)(tok0 + s0 - WIN), (int)bco);
        mbar_arrive_expect_tx(&S.bar_g, 32768u);
        tma_load_4d(sm + lG, &tmG, &S.bar_g, 0, (int)kv, (int)(tok0 + s0), (int)bco);
        local_load(sm + lV, &tmV, &S.bar_v, kv, tok0 + s0 - WIN, bco);
        k_out = v_out = g_out = true;
    }
    tc_fence_before();
    __syncthreads();
    uint32_t ph_k = 0, ph_v = 0, ph_g = 0, ph_u = 0, ph_h = 0;
    float lam_tot = 0.0f;
    bool ok = true;

    for (int64_t c = 0; c < nsteps; ++c) {
        const int64_t t0 = s0 + c * LT;
        const int n = (int)min64(LT, s1 - t0);
        const bool more = c + 1 < nsteps;
        // (1) U_k = k Wf for the 128 delayed keys of the step
        ok = local_wait(&S.bar_k, ph_k, S, hdr, 20);
        if (!ok) break;
        if (zero_pre && c == 0) {
            // rows t < WIN - s0 of both 64-column halves (the swizzle permutes chunks within
            // a row, so whole rows are zeroed)
            const int nz = (int)(WIN - s0) * 2 * 8;
            for (int e = tid; e < nz; e += NL) {
                const int r = e >> 4, kb = (e >> 3) & 1, ch = e & 7;
                st_shared_v4(base + lK + kb * 16384 + r * 128 + ch * 16, 0u, 0u, 0u, 0u);
            }
            fence_async_smem();
            __syncthreads();
        }
        if (tid == 0) {
            k_out = false;
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t koff = ((j >> 2) * 16384 + (j & 3) * 32) >> 4;
                mma_bf16(tb + cUl, dK + koff, dW + ((j * 2048) >> 4), idesc_bf16(128, 64, false, true),
                         j > 0);
            }
            mma_commit(&S.bar_u);
            mma_out = true;
        }
        // (2) gates: four threads per feature, 32 tokens each; decay of each token's key to the
        //     step end, e^{b_last - b_t} (at most 1), and of the old state, e^{b_last}.  Both are
        //     products of Gamma = 1 / (1 + e^{-g}): suffix products inside the thread's quarter
        //     times the later quarters' products.  The step's log-decay (for the records) comes
        //     from the quarter products renormalised every 4 tokens, one logarithm per thread.
        ok = local_wait(&S.bar_g, ph_g, S, hdr, 21);
        if (!ok) break;
        if (tid == 0) g_out = false;
        {
            const int gf = tid & (DF - 1), gq = tid >> 7;
            const __nv_bfloat16* sg = (const __nv_bfloat16*)(sm + lG);
            float suf[32];       // prod_{s = t+1 .. quarter end} Gamma_s
            float sp = 1.0f;     // running suffix product
            float mq = 1.0f;     // the same product, renormalised: mq 2^{eq}
            int eq = 0;
#pragma unroll
            for (int j = 31; j >= 0; --j) {
                const int tt = 32 * gq + j;
                const float gam =
                    tt < n ? rcpf(1.0f + ex2f(-__bfloat162float(sg[tt * DF + gf]) * kLog2e)) : 1.0f;
                suf[j] = sp;
                sp *= gam;
                mq *= gam;
                if ((j & 3) == 0) {
                    int e;
                    mq = frexpf(mq, &e);
                    eq += e;
                }
            }
            gpart[gq * DF + gf] = sp;                                // the quarter's product
            zq[gq * DF + gf] = (__log2f(mq) + (float)eq) * kLn2;     // and its logarithm
            __syncthreads();
            const float q1 = gpart[DF + gf], q2 = gpart[2 * DF + gf], q3 = gpart[3 * DF + gf];
            const float later = gq == 3 ? 1.0f : gq == 2 ? q3 : gq == 1 ? q2 * q3 : (q1 * q2) * q3;
            // kept in fp32: the state records feed the gate gradient, a difference of two
            // nearly equal sums that bf16 weights would not cancel consistently
            float* Ek = (float*)(sm + lE);
#pragma unroll
            for (int j = 0; j < 32; ++j) Ek[(32 * gq + j) * EKR + gf] = suf[j] * later;
            // masked decay reading: each delayed key enters scaled by the product of the w
            // gates it saw in the window, e^{kd}, folded into its decay factor; the loads of
            // each batch of the thread's 32 rows are issued before its first product
            // (kd = 0: no factor)
            if (KEYF) {
                constexpr int KB = 16;
                const int64_t kstride = p.Hkv * DF;
                const float* kcol = a.kdec + (row0 * p.Hkv + kv) * DF + gf;
#pragma unroll 1
                for (int j0 = 0; j0 < 32; j0 += KB) {
                    float kdl[KB];
#pragma unroll
                    for (int j = 0; j < KB; ++j) {
                        const int64_t key = t0 + 32 * gq + j0 + j - WIN;
                        kdl[j] = key >= 0 && 32 * gq + j0 + j < n ? kcol[key * kstride] : 0.0f;
                    }
#pragma unroll
                    for (int j = 0; j < KB; ++j) Ek[(32 * gq + j0 + j) * EKR + gf] *= __expf(kdl[j]);
                }
                // the next step's factors, into L2 while this step computes
#pragma unroll 8
                for (int j = 0; j < 32; ++j) {
                    const int64_t key = t0 + LT + 32 * gq + j - WIN;
                    if (key >= 0 && key + WIN < s1) prefetch_l2(kcol + key * kstride);
                }
            }
            if (gq == 0) {
                S.el[gf] = gpart[gf] * ((q1 * q2) * q3);
                lam_tot += (zq[gf] + zq[DF + gf]) + (zq[2 * DF + gf] + zq[3 * DF + gf]);
            }
        }
        __syncthreads();
        // the gate tile is consumed: the next step's gates start loading
        if (tid == 0 && more) {
            mbar_arrive_expect_tx(&S.bar_g, 32768u);
            tma_load_4d(sm + lG, &tmG, &S.bar_g, 0, (int)kv, (int)(tok0 + t0 + LT), (int)bco);
            g_out = true;
        }
        // (3) decay the state by e^{b_last} (lane = feature, 32 columns per part)
        {
            float v[32];
            tmem_ld32(tb + lane_off + cHl + 32 * part, v);
            tmem_wait_ld();
            const float el = S.el[row];
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] *= el;
            tmem_st32(tb + lane_off + cHl + 32 * part, v);
            tmem_wait_st();
        }
        // (4) phi of the delayed keys (lane = key): parts 0, 1 softmax(+u) over features
        //     [0, 64), parts 2, 3 softmax(-u) over [64, 128); k~ = phi e^{b_last - b_t}
        ok = local_wait(&S.bar_u, ph_u, S, hdr, 22);
        if (!ok) break;
        tc_fence_after();
        if (tid == 0) {
            mma_out = false;
            // the key tile is consumed: the next step's keys start loading
            if (more) {
                local_load(sm + lK, &tmK, &S.bar_k, kv, tok0 + t0 + LT - WIN, bco);
                k_out = true;
            }
        }
        {
            const int t = row, sib = part ^ 1;
            float uv[32];
            tmem_ld32(tb + lane_off + cUl + 32 * (part & 1), uv);
            tmem_wait_ld();
            float uext = -INFINITY;
            if (part < 2) {
#pragma unroll
                for (int k = 0; k < 32; ++k) uext = fmaxf(uext, uv[k]);
            } else {
#pragma unroll
                for (int k = 0; k < 32; ++k) uext = fmaxf(uext, -uv[k]);
            }
            xum[part * 128 + t] = uext;
            quad_sync(quad);
            const float f2 = part < 2 ? kLog2e : -kLog2e;
            const float cst = -fmaxf(xum[part * 128 + t], xum[sib * 128 + t]) * kLog2e;
            float usum = 0.0f;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                uv[k] = ex2f(fmaf(uv[k], f2, cst));
                usum += uv[k];
            }
            xus[part * 128 + t] = usum;
            quad_sync(quad);
            const bool dvalid = (t0 + t - WIN >= 0) && (t < n);
            const float inv = dvalid ? 1.0f / (xus[part * 128 + t] + xus[sib * 128 + t]) : 0.0f;
            // high and low bf16 parts: the state these records start segments from must carry
            // fp32-like precision (the backward differentiates through it); the low parts go
            // over the decay table once every thread has read its rows of it
            uint32_t lo[16];
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                const int f0 = 32 * part + 8 * ch;
                const float4* ep = reinterpret_cast<const float4*>(sm + lE + (size_t)(t * EKR + f0) * 4u);
                const float4 e0 = ep[0], e1 = ep[1];
                const float ek[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
                float kv8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) kv8[e] = uv[8 * ch + e] * inv * ek[e];
                uint32_t hi[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) split2(kv8[2 * e], kv8[2 * e + 1], hi[e], lo[4 * ch + e]);
                const uint32_t o = (part >> 1) * 16384 + sw128(t, 4 * (part & 1) + ch);
                st_shared_v4(base + lKu + o, hi[0], hi[1], hi[2], hi[3]);
            }
            __syncthreads();
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                const uint32_t o = (part >> 1) * 16384 + sw128(t, 4 * (part & 1) + ch);
                st_shared_v4(base + lKul + o, lo[4 * ch], lo[4 * ch + 1], lo[4 * ch + 2], lo[4 * ch + 3]);
            }
        }
        if (zero_pre && c == 0) {
            // the value rows before the sequence start, as for the keys (every thread waits
            // for the tile here; the issuing thread's wait below then returns at once)
            mbar_wait(&S.bar_v, 0u, kTimeout);
            const int nz = (int)(WIN - s0) * 2 * 8;
            for (int e = tid; e < nz; e += NL) {
                const int r = e >> 4, kb = (e >> 3) & 1, ch = e & 7;
                st_shared_v4(base + lV + kb * 16384 + r * 128 + ch * 16, 0u, 0u, 0u, 0u);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // (5) H += k~^T v on the tensor cores while the threads sum z
        if (tid == 0) {
            if (!mbar_wait(&S.bar_v, ph_v, kTimeout)) {
                S.abort = 1;
                report(hdr, LIZARD_ERR_TIMEOUT, 23);
            } else {
                ph_v ^= 1u;
                v_out = false;
                tc_fence_after();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    mma_bf16(tb + cHl, dKu + ((j * 2048) >> 4), dV + ((j * 2048) >> 4),
                             idesc_bf16(128, 128, true, true), 1);
                    mma_bf16(tb + cHl, dKul + ((j * 2048) >> 4), dV + ((j * 2048) >> 4),
                             idesc_bf16(128, 128, true, true), 1);
                }
                mma_commit(&S.bar_h);
                mma_out = true;
            }
        }
        {
            // z <- e^{b_last} z + sum_t k~_t, from the bf16 tile the MMA reads
            const int f = tid & (DF - 1), gq = tid >> 7;
            const __nv_bfloat16* ku = (const __nv_bfloat16*)(sm + lKu);
            const __nv_bfloat16* kul = (const __nv_bfloat16*)(sm + lKul);
            float zs[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // four chains: the loads overlap
#pragma unroll
            for (int t = 32 * gq; t < 32 * gq + 32; ++t) {
                const uint32_t off = ((f >> 6) * 16384 + sw128(t, (f & 63) >> 3) + (f & 7) * 2) / 2;
                zs[t & 3] += __bfloat162float(ku[off]) + __bfloat162float(kul[off]);
            }
            zq[gq * DF + f] = (zs[0] + zs[1]) + (zs[2] + zs[3]);
        }
        __syncthreads();
        if (tid < DF)
            S.z[tid] = fmaf(S.el[tid], S.z[tid], (zq[tid] + zq[DF + tid]) + (zq[2 * DF + tid] + zq[3 * DF + tid]));
        ok = local_wait(&S.bar_h, ph_h, S, hdr, 24);
        if (!ok) break;
        tc_fence_after();
        if (tid == 0) {
            mma_out = false;
            // values and k~ are consumed: the next step's values start loading
            if (more) {
                local_load(sm + lV, &tmV, &S.bar_v, kv, tok0 + t0 + LT - WIN, bco);
                v_out = true;
            }
        }
    }

    if (ok) {
        float* r = a.seg + ((size_t)seg * (size_t)U + (size_t)unit) * p.rec_floats;
        float v[32];
        tmem_ld32(tb + lane_off + cHl + 32 * part, v);
        tmem_wait_ld();
        // through the (now idle) key and value tiles, then coalesced to the record
        staged_row_write(sm + lK, row, part, v);
        __syncthreads();
        stage_record_out(r, sm + lK);
        if (tid < DF) {
            r[DF * DH + tid] = S.z[tid];
            r[DF * DH + DF + tid] = lam_tot;
        }
    } else if (tid == 0) {
        // let copies and MMAs still in flight land before the CTA exits
        if (mma_out) {
            mma_commit(&S.bar_fin);
            mbar_wait(&S.bar_fin, 0, kTimeout);
        }
        if (k_out) mbar_wait(&S.bar_k, ph_k, kTimeout);
        if (g_out) mbar_wait(&S.bar_g, ph_g, kTimeout);
        if (v_out) mbar_wait(&S.bar_v, ph_v, kTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 256);
    }
}

// Segment pass (fwd_tc_local) over every segment but the last, then the exclusive scan:
// a.seg receives the state each segment starts from.
cudaError_t launch_local_and_scan(const Plan& p, const FwdArgs& a, const CUtensorMap& mw,
                                  cudaStream_t s) {
    // packed sequences: maps over all T rows, batch extent 1
    const cuuint64_t B = p.cu != nullptr ? 1 : (cuuint64_t)p.B,
                     L = p.cu != nullptr ? (cuuint64_t)p.T : (cuuint64_t)p.L,
                     Hkv = (cuuint64_t)p.Hkv;
    const unsigned U = (unsigned)(p.B * p.Hkv);
    // 128-token tiles of the delayed keys, values and gates
    alignas(64) CUtensorMap lk, lv, lg;
    {
        const cuuint64_t dims[4] = {DH, Hkv, L, B};
        const cuuint64_t str[3] = {DH * 2, Hkv * DH * 2, L * Hkv * DH * 2};
        const cuuint32_t box[4] = {64, 1, LT, 1};
        if (!make_map(&lk, a.k, 4, dims, str, box)) return cudaErrorInvalidValue;
        if (!make_map(&lv, a.v, 4, dims, str, box)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[4] = {DF, Hkv, L, B};
        const cuuint64_t str[3] = {DF * 2, Hkv * DF * 2, L * Hkv * DF * 2};
        const cuuint32_t box[4] = {DF, 1, LT, 1};
        if (!make_map(&lg, a.g, 4, dims, str, box, false)) return cudaErrorInvalidValue;
    }
    auto local = a.kdec != nullptr ? fwd_tc_local<true> : fwd_tc_local<false>;
    cudaError_t e = cudaFuncSetAttribute(local, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kLocalSmem);
    if (e != cudaSuccess) return e;
    local<<<dim3(U, (unsigned)(p.P - 1)), NL, kLocalSmem, s>>>(lk, lv, mw, lg, p, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_seg_scan(p, a.seg, s, true);
}

bool make_wf_map(CUtensorMap* mw, const void* Wf, int64_t Hkv) {
    const cuuint64_t dims[3] = {DF / 2, DH, (cuuint64_t)Hkv};
    const cuuint64_t str[2] = {(DF / 2) * 2, DH * (DF / 2) * 2};
    const cuuint32_t box[3] = {DF / 2, DH, 1};
    return make_map(mw, Wf, 3, dims, str, box);
}

}  // namespace

bool fwd_tc_supported(const Plan& p) {
    return p.dtype == LIZARD_BF16 && p.d == DH && p.D == DF && p.G == GQ && p.w == WIN &&
           p.M <= MMAX && p.L < ((int64_t)1 << 30) && p.T < ((int64_t)1 << 30) &&
           encode_fn() != nullptr;
}

cudaError_t launch_fwd_states_tc(const Plan& p, const FwdArgs& a, cudaStream_t s) {
    if (p.P <= 1) return cudaSuccess;
    alignas(64) CUtensorMap mw;
    if (!make_wf_map(&mw, a.Wf, p.Hkv)) return cudaErrorInvalidValue;
    return launch_local_and_scan(p, a, mw, s);
}

// Segments are cut so that the last wave of (batch, KV head, segment) CTAs is as full as the
// others: a second, mostly empty wave would cost a whole segment's walk.
//
// With few segments the segment pass (one CTA per unit and segment but the last) would leave
// SMs idle, so its records are cut rec_step times finer while one wave still holds them: the
// scan then yields the state at every finer boundary and the main walk reads every
// rec_step-th record.
void fwd_tc_plan(Plan* p) {
    p->rec_step = 1;
    if (p->cu != nullptr) return;  // packed sequences come with their segments cut
    plan_segments_waves(p, 152);
    if (p->P <= 1) return;
    const int64_t U = p->B * p->Hkv;
    for (int64_t k = 2; k <= 8; ++k) {
        if (U * k * (p->P - 1) > 152 || k * (p->P - 1) + 1 > p->Pmax) break;
        if (p->seg_chunks % k == 0) p->rec_step = k;
    }
}

cudaError_t launch_fwd_tc(const Plan& p0, const FwdArgs& a, cudaStream_t s) {
    Plan p = p0;
    fwd_tc_plan(&p);
    alignas(64) CUtensorMap mq, mk, mv, mw, my;
    // packed sequences: maps over all T rows, batch extent 1
    const cuuint64_t B = p.cu != nullptr ? 1 : (cuuint64_t)p.B,
                     L = p.cu != nullptr ? (cuuint64_t)p.T : (cuuint64_t)p.L,
                     Hq = (cuuint64_t)p.Hq, Hkv = (cuuint64_t)p.Hkv;
    {
        const cuuint64_t dims[4] = {DH, Hq, L, B};
        const cuuint64_t str[3] = {DH * 2, Hq * DH * 2, L * Hq * DH * 2};
        const cuuint32_t box[4] = {64, GQ, CT, 1};
        if (!make_map(&mq, a.q, 4, dims, str, box)) return cudaErrorInvalidValue;
        if (!make_map(&my, a.y, 4, dims, str, box)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[4] = {DH, Hkv, L, B};
        const cuuint64_t str[3] = {DH * 2, Hkv * DH * 2, L * Hkv * DH * 2};
        const cuuint32_t box[4] = {64, 1, CT, 1};
        if (!make_map(&mk, a.k, 4, dims, str, box)) return cudaErrorInvalidValue;
        if (!make_map(&mv, a.v, 4, dims, str, box)) return cudaErrorInvalidValue;
    }
    alignas(64) CUtensorMap mg;
    {
        const cuuint64_t dims[4] = {DF, Hkv, L, B};
        const cuuint64_t str[3] = {DF * 2, Hkv * DF * 2, L * Hkv * DF * 2};
        const cuuint32_t box[4] = {DF, 1, CT, 1};
        if (!make_map(&mg, a.g, 4, dims, str, box, false)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {DF / 2, DH, Hkv};
        const cuuint64_t str[2] = {(DF / 2) * 2, DH * (DF / 2) * 2};
        const cuuint32_t box[3] = {DF / 2, DH, 1};
        if (!make_map(&mw, a.Wf, 3, dims, str, box)) return cudaErrorInvalidValue;
    }
    cudaError_t e;
    auto walk = a.kdec != nullptr ? fwd_tc_kernel<true> : fwd_tc_kernel<false>;
    e = cudaFuncSetAttribute(walk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const unsigned U = (unsigned)(p.B * p.Hkv);
    if (p.P > 1) {
        // the segment pass and the scan over rec_step finer cuts of every segment but the last
        Plan pl = p;
        pl.seg_chunks = p.seg_chunks / p.rec_step;
        pl.seg_len = pl.seg_chunks * kChunk;
        pl.P = p.rec_step * (p.P - 1) + 1;
        pl.rec_step = 1;
        e = launch_local_and_scan(pl, a, mw, s);
        if (e != cudaSuccess) return e;
    }
    if (a.ev_before) cudaEventRecord(a.ev_before, s);
    if (p.P > 1 && a.ev_before == nullptr)  // starts while the scan finishes
        e = launch_dependent(walk, dim3(U, (unsigned)p.P), dim3(NT), kSmemBytes, s, mq, mk, mv,
                             mw, mg, my, p, a);
    else
        walk<<<dim3(U, (unsigned)p.P), NT, kSmemBytes, s>>>(mq, mk, mv, mw, mg, my, p, a);
    if (a.ev_after) cudaEventRecord(a.ev_after, s);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // segments handed over at a strongly closed step are finished by the exact walk
    return launch_fwd_tail(p, a, s);
}

}  // namespace lz
