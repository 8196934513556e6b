// Backward of the Lizard token mixer (exact gradient of the forward; the pages give no
// backward, so this is the adjoint of the definition).  SIMT, fp32 arithmetic.
//
// With a_i = 1/den_i = e^{-lse_i}, delta_i = dy_i . y_i and g^_i = a_i [dy_i, -delta_i],
// the pieces are (Lizard summary, gist.science/ko/paper/2507.09025, sec. 2-A and 2-C):
//   window (sec. 2-A-2): p_ij = e^{s q_i.k_j - lse_i}, ds_ij = p_ij (dy_i.v_j - delta_i),
//       dq_i += s sum_j ds_ij k_j, dk_j += s sum_i ds_ij q_i, dv_j += sum_i p_ij dy_i;
//   sinks: dt_hm = -e^{t_hm} sum_i a_i delta_i;
//   state (sec. 2-A-1): with k'_t = k_{t-w}, v^'_t = [v_{t-w}, 1] and the pair weight
//       e^{B_i - B_t} (B = cumulative log-sigmoid gate, t <= i):
//       dphi(q_i)_f  = sum_t e^{B_if - B_tf} phi(k'_t)_f (v^'_t . g^_i)
//       dphi(k'_t)_f = sum_i e^{B_if - B_tf} phi(q_i)_f (v^'_t . g^_i)
//       dv'_t        = sum_i (sum_f e^{B_if - B_tf} phi(q_i)_f phi(k'_t)_f) dy_i a_i
//       dB_s = phi(q_s) (.) dphi(q_s) - phi(k'_s) (.) dphi(k'_s),
//       dlambda_u = sum_{s >= u} dB_s, dg = dlambda (1 - sigmoid(g));
//   feature map (sec. 2-C): du = p (dp - p.dp) - n (dn - n.dn), dx = Wf du, dWf += x du^T.
//
// Launch sequence: forward segment states (segment pass + scan) -> forward-direction walk
// (dq, phi(q)-side of dB, dWf/dsinks partials) -> reverse segment pass + reverse scan of
// the state adjoint -> reverse-direction walk (state parts of dk, dv, phi(k)-side of dB,
// reverse cumulative sum of dB inside each segment, dWf partials) -> key-centric window
// pass (adds the window parts of dk, dv) -> dg -> fixed-order reductions of dWf, dsinks.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "simt.cuh"

namespace lz {
namespace {

using simt::NT;
constexpr int TS = 16;  // tokens per step of the two walks
constexpr int LPR = 16; // lanes per row
constexpr int KB = 16;  // window keys per tile in the query-side walk

// Workspace regions (floats, each 64-float aligned)
struct BwdWs {
    size_t fwd_rec, rev_rec, dB, tot, dW, dt, rows, flags;
    size_t gl, kd, kk, kt;  // decay readings: moved gates (LAGGED); key log products, their gate
                            // terms and the terms' chunk totals (MASKED)
    size_t total;
};

inline size_t al64(size_t x) { return (x + 63) & ~(size_t)63; }

BwdWs bwd_layout(const Plan& p) {
    BwdWs w;
    const size_t U = (size_t)(p.B * p.Hkv);
    size_t off = kHeaderBytes / sizeof(float);
    w.fwd_rec = off;
    off += al64((size_t)p.Pmax * U * p.rec_floats);
    w.rev_rec = off;
    off += al64((size_t)p.Pmax * U * p.rec_floats);
    w.dB = off;
    off += al64((size_t)(p.B * p.L * p.Hkv) * (size_t)p.D);
    w.tot = off;
    off += al64((size_t)p.Pmax * U * (size_t)p.D);
    w.dW = off;
    off += al64((size_t)2 * p.Pmax * U * (size_t)(p.d * (p.D / 2)));
    w.dt = off;
    off += al64((size_t)p.Pmax * U * (size_t)p.G);
    w.rows = off;  // per query row: a = e^{-lse}, delta = dy . y   [2][B*L*Hq]
    off += al64((size_t)2 * (size_t)(p.B * p.L * p.Hq));
    w.flags = off;  // per (segment, unit): 1 if its gates close too hard for the factored walks
    off += al64((size_t)p.Pmax * U);
    const size_t ng = (size_t)(p.B * p.L * p.Hkv) * (size_t)p.D;
    w.gl = off;  // LAGGED: g moved w tokens later, in the input's dtype
    if (p.decay == LIZARD_DECAY_LAGGED) off += al64((ng * (p.dtype == LIZARD_F32 ? 4 : 2) + 3) / 4);
    w.kd = off;  // MASKED: log product of the w gates after each key
    if (p.decay == LIZARD_DECAY_MASKED) off += al64(ng);
    w.kk = off;  // MASKED: phi(k') (.) dphi(k') of each key, at the key's own row
    if (p.decay == LIZARD_DECAY_MASKED) off += al64(ng);
    w.kt = off;  // MASKED: chunk totals of those terms (their suffix sums)
    if (p.decay == LIZARD_DECAY_MASKED) off += al64(key_suffix_scratch_floats(p));
    w.total = off * sizeof(float);
    return w;
}

// Shared-memory layout of the two walks (floats).  Rows that are read across lanes are
// padded by one float.
template <int DH, int DF>
struct BLay {
    static constexpr int PF = DF + 1, PH = DH + 1, H2 = DF / 2, PW = DF / 2 + 1;
    static constexpr int oH = 0;                    // state or its adjoint [DF][PH]
    static constexpr int oz = oH + DF * PH;          // [DF]
    static constexpr int oW = oz + DF;              // Wf [DH][PW]
    static constexpr int ob = oW + DH * PW;         // cumulative log-gates [TS][PF]
    static constexpr int ophk = ob + TS * PF;       // phi(k') [TS][PF]
    static constexpr int ov = ophk + TS * PF;       // v' [TS][PH]
    static constexpr int oq = ov + TS * PH;         // raw x rows [TS][PH]
    static constexpr int ophq = oq + TS * PH;       // phi(q) [TS][PF]
    static constexpr int odp = ophq + TS * PF;      // dphi / du [TS][PF]
    static constexpr int ody = odp + TS * PF;       // dy [TS][PH]
    static constexpr int oA = ody + TS * PH;        // pair scalars [TS][TS+1]
    static constexpr int oA2 = oA + TS * (TS + 1);  // second pair matrix [TS][TS+1]
    static constexpr int orow = oA2 + TS * (TS + 1);  // a_i, delta_i, lse_i [3][TS]
    static constexpr int otile = orow + 3 * TS;     // window key/value tiles [2][KB][PH], ds [TS][KB]
                                                    // (reverse walk: decay tables [2][TS][PF], [2][DF])
    static constexpr int ntile = 2 * KB * PH + TS * KB > 2 * TS * PF + 2 * DF
                                     ? 2 * KB * PH + TS * KB
                                     : 2 * TS * PF + 2 * DF;
    static constexpr int total = otile + ntile;
    static constexpr size_t bytes = sizeof(float) * (size_t)total;
};

// phi rows with a padded Wf (row stride PW); rows outside [rlo, rhi) are zero.
template <int DH, int DF, bool FAST>
__device__ __forceinline__ void phi_rows_p(const float* sx, const float* sW, float* sout, int rlo,
                                           int rhi) {
    constexpr int H = DF / 2, PH = DH + 1, PF = DF + 1, PW = DF / 2 + 1, NJ = H / LPR;
    const int r = threadIdx.x / LPR, sub = threadIdx.x % LPR;
    float u[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) u[j] = 0.0f;
    const float* x = sx + r * PH;
    for (int c = 0; c < DH; ++c) {
        const float xc = x[c];
#pragma unroll
        for (int j = 0; j < NJ; ++j) u[j] = fmaf(xc, sW[c * PW + sub + LPR * j], u[j]);
    }
    float mx = u[0], mn = u[0];
#pragma unroll
    for (int j = 1; j < NJ; ++j) {
        mx = fmaxf(mx, u[j]);
        mn = fminf(mn, u[j]);
    }
#pragma unroll
    for (int o = 1; o < LPR; o <<= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    }
    float ep[NJ], en[NJ], sp = 0.0f, sn = 0.0f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        ep[j] = ex<FAST>(u[j] - mx);
        en[j] = ex<FAST>(mn - u[j]);
        sp += ep[j];
        sn += en[j];
    }
#pragma unroll
    for (int o = 1; o < LPR; o <<= 1) {
        sp += __shfl_xor_sync(0xffffffffu, sp, o);
        sn += __shfl_xor_sync(0xffffffffu, sn, o);
    }
    const bool valid = r >= rlo && r < rhi;
    const float ip = valid ? 1.0f / sp : 0.0f, in = valid ? 1.0f / sn : 0.0f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        sout[r * PF + sub + LPR * j] = ep[j] * ip;
        sout[r * PF + H + sub + LPR * j] = en[j] * in;
    }
}

// Feature-map backward of TS rows: from phi (sphi) and dphi (sdp), du[r][f] (f < D/2) is
// written into sdp in place.  Eight lanes per row.
template <int DF>
__device__ __forceinline__ void phi_backward_rows(const float* sphi, float* sdp) {
    constexpr int H = DF / 2, PF = DF + 1, NJ = H / LPR;
    const int r = threadIdx.x / LPR, sub = threadIdx.x % LPR;
    float sp = 0.0f, sn = 0.0f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const int f = sub + LPR * j;
        sp = fmaf(sphi[r * PF + f], sdp[r * PF + f], sp);
        sn = fmaf(sphi[r * PF + H + f], sdp[r * PF + H + f], sn);
    }
#pragma unroll
    for (int o = 1; o < LPR; o <<= 1) {
        sp += __shfl_xor_sync(0xffffffffu, sp, o);
        sn += __shfl_xor_sync(0xffffffffu, sn, o);
    }
    float du[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const int f = sub + LPR * j;
        du[j] = sphi[r * PF + f] * (sdp[r * PF + f] - sp) -
                sphi[r * PF + H + f] * (sdp[r * PF + H + f] - sn);
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < NJ; ++j) sdp[r * PF + sub + LPR * j] = du[j];
}

template <typename T, int DH>
__device__ __forceinline__ void load_rows_p(const T* x, int64_t b, int64_t L, int64_t Hx,
                                            int64_t hx, int64_t tok0, int rlo, int rhi, float* s) {
    constexpr int PH = DH + 1;
    for (int e = threadIdx.x; e < TS * DH; e += NT) {
        const int t = e / DH, c = e % DH;
        float val = 0.0f;
        if (t >= rlo && t < rhi) val = ld(x + ((b * L + tok0 + t) * Hx + hx) * DH + c);
        s[t * PH + c] = val;
    }
}

// a_i = e^{-lse_i}, delta_i = dy_i . y_i, lse_i for the n valid rows of one head, from the
// per-row table the first backward kernel fills.
__device__ __forceinline__ void row_stats(const BwdArgs& a, const Plan& p, const BwdWs& ws,
                                          int64_t b, int64_t h, int64_t i0, int n, float* srow) {
    const int r = threadIdx.x;
    if (r < TS) {
        const int64_t idx = (b * p.L + i0 + r) * p.Hq + h;
        const int64_t nrow = p.B * p.L * p.Hq;
        const float* rows = (const float*)a.ws + ws.rows;
        srow[r] = r < n ? rows[idx] : 0.0f;
        srow[TS + r] = r < n ? rows[nrow + idx] : 0.0f;
        srow[2 * TS + r] = r < n ? a.lse[idx] : 0.0f;
    }
}

// Per query row: a = e^{-lse}, delta = dy . y (one warp per row, fixed order).
template <typename T, int DH>
__global__ void bwd_row_table(Plan p, BwdArgs a, BwdWs ws) {
    const int64_t nrow = p.B * p.L * p.Hq;
    const int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= nrow) return;
    const T* yr = (const T*)a.y + r * DH;
    const T* dr = (const T*)a.dy + r * DH;
    float dl = 0.0f;
    for (int c = lane; c < DH; c += 32) dl = fmaf(ld(yr + c), ld(dr + c), dl);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dl += __shfl_xor_sync(0xffffffffu, dl, o);
    if (lane == 0) {
        float* rows = (float*)a.ws + ws.rows;
        rows[r] = expf(-a.lse[r]);
        rows[nrow + r] = dl;
    }
}

// bf16, d = 128: 16 lanes per row (8 elements each, 16-byte loads), 8 rows per warp with every
// load of the warp issued before the first use, so each warp keeps 4 KB in flight.
constexpr int kRowsPerWarp = 8;
__global__ void bwd_row_table_bf16(Plan p, BwdArgs a, BwdWs ws) {
    const int64_t nrow = p.B * p.L * p.Hq;
    const int64_t r0 = ((int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5)) * kRowsPerWarp;
    const int lane = threadIdx.x & 31, half = lane >> 4, sub = lane & 15;
    uint4 yv[kRowsPerWarp / 2], dv[kRowsPerWarp / 2];
    float ls[kRowsPerWarp / 2];
#pragma unroll
    for (int k = 0; k < kRowsPerWarp / 2; ++k) {
        const int64_t r = r0 + 2 * k + half;
        const bool in = r < nrow;
        yv[k] = in ? reinterpret_cast<const uint4*>((const __nv_bfloat16*)a.y + r * 128)[sub] : make_uint4(0u, 0u, 0u, 0u);
        dv[k] = in ? reinterpret_cast<const uint4*>((const __nv_bfloat16*)a.dy + r * 128)[sub] : make_uint4(0u, 0u, 0u, 0u);
        ls[k] = in && sub == 0 ? a.lse[r] : 0.0f;
    }
    float* rows = (float*)a.ws + ws.rows;
#pragma unroll
    for (int k = 0; k < kRowsPerWarp / 2; ++k) {
        const uint32_t yw[4] = {yv[k].x, yv[k].y, yv[k].z, yv[k].w};
        const uint32_t dw[4] = {dv[k].x, dv[k].y, dv[k].z, dv[k].w};
        float dl = 0.0f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            dl = fmaf(__uint_as_float(yw[e] << 16), __uint_as_float(dw[e] << 16), dl);
            dl = fmaf(__uint_as_float(yw[e] & 0xFFFF0000u), __uint_as_float(dw[e] & 0xFFFF0000u), dl);
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) dl += __shfl_xor_sync(0xffffffffu, dl, o);
        const int64_t r = r0 + 2 * k + half;
        if (sub == 0 && r < nrow) {
            rows[r] = expf(-ls[k]);
            rows[nrow + r] = dl;
        }
    }
}

// sb[t][f] = sum_{s<=t} log sigmoid(g_{i0+s, f}) over TS rows (rows >= n add 0).
template <typename T, int DF, bool FAST>
__device__ __forceinline__ void gates_cumsum_b(const T* g, int64_t b, int64_t L, int64_t Hkv,
                                               int64_t kv, int64_t i0, int n, float* sb) {
    constexpr int PF = DF + 1;
    for (int e = threadIdx.x; e < TS * DF; e += NT) {
        const int t = e / DF, f = e % DF;
        float lam = 0.0f;
        if (t < n) lam = log_sigmoid<FAST>(ld(g + ((b * L + i0 + t) * Hkv + kv) * DF + f));
        sb[t * PF + f] = lam;
    }
    __syncthreads();
    if (threadIdx.x < DF) {
        const int f = threadIdx.x;
        float acc = 0.0f;
        for (int t = 0; t < TS; ++t) {
            acc += sb[t * PF + f];
            sb[t * PF + f] = acc;
        }
    }
    __syncthreads();
}

// Forward-direction state update over one step (augmented with z).  Overwrites sphk.
template <int DH, int DF, bool FAST>
__device__ __forceinline__ void state_step(float* sH, float* sz, float* sphk, const float* sv,
                                           const float* sb) {
    constexpr int PF = DF + 1, PH = DH + 1;
    for (int e = threadIdx.x; e < TS * DF; e += NT) {
        const int t = e / DF, f = e % DF;
        sphk[t * PF + f] *= ex<FAST>(sb[(TS - 1) * PF + f] - sb[t * PF + f]);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < DF * DH; e += NT) {
        const int f = e / DH, c = e % DH;
        float acc = ex<FAST>(sb[(TS - 1) * PF + f]) * sH[f * PH + c];
        for (int t = 0; t < TS; ++t) acc = fmaf(sphk[t * PF + f], sv[t * PH + c], acc);
        sH[f * PH + c] = acc;
    }
    if (threadIdx.x < DF) {
        const int f = threadIdx.x;
        float acc = ex<FAST>(sb[(TS - 1) * PF + f]) * sz[f];
        for (int t = 0; t < TS; ++t) acc += sphk[t * PF + f];
        sz[f] = acc;
    }
    __syncthreads();
}

// Adjoint accumulation: [dH | dz] += sum_t (e^{b_t} phq_t a_t) [dy_t, -delta_t].
// Overwrites sphq with the scaled rows.  Each thread accumulates a block of DF/8 features x
// DH/32 columns in registers (columns lane + 32 k, features of its warp), so a step reads
// each scaled feature once per warp and each dy value once per thread.
template <int DH, int DF, bool FAST>
__device__ __forceinline__ void adjoint_add(float* sH, float* sz, float* sphq, const float* sdy,
                                            const float* sb, const float* srow, int n,
                                            const float* ser = nullptr) {
    constexpr int PF = DF + 1, PH = DH + 1;
    constexpr int NWARP = NT / 32, FB = DF / NWARP, NCC = DH / 32;
    // rows become e^{b_t} phi(q_t) a_t; when ser is given the rows already carry e^{b_t - r}
    // and ser[f] = e^{r_f} completes the factor
    for (int e = threadIdx.x; e < TS * DF; e += NT) {
        const int t = e / DF, f = e % DF;
        sphq[t * PF + f] *= (ser ? ser[f] : ex<FAST>(sb[t * PF + f])) * srow[t];
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, wf = (threadIdx.x >> 5) * FB;
    float acc[FB][NCC];
#pragma unroll
    for (int j = 0; j < FB; ++j)
#pragma unroll
        for (int k = 0; k < NCC; ++k) acc[j][k] = sH[(wf + j) * PH + lane + 32 * k];
    for (int t = 0; t < n; ++t) {
        float dyv[NCC];
#pragma unroll
        for (int k = 0; k < NCC; ++k) dyv[k] = sdy[t * PH + lane + 32 * k];
#pragma unroll
        for (int j = 0; j < FB; ++j) {
            const float ph = sphq[t * PF + wf + j];
#pragma unroll
            for (int k = 0; k < NCC; ++k) acc[j][k] = fmaf(ph, dyv[k], acc[j][k]);
        }
    }
#pragma unroll
    for (int j = 0; j < FB; ++j)
#pragma unroll
        for (int k = 0; k < NCC; ++k) sH[(wf + j) * PH + lane + 32 * k] = acc[j][k];
    if (threadIdx.x < DF) {
        float za = sz[threadIdx.x];
        for (int t = 0; t < n; ++t) za = fmaf(-sphq[t * PF + threadIdx.x], srow[TS + t], za);
        sz[threadIdx.x] = za;
    }
    __syncthreads();
}

// ---------------------------------------------------------------------------------------
// Forward-direction walk: dq (state and window parts), phi(q)-side of dB, partials.
// One CTA per (batch, KV head, segment); the G query heads are walked in turn.
template <typename T, int DH, int DF, bool FAST>
__global__ void __launch_bounds__(NT, 1) bwd_forward_walk(Plan p, BwdArgs a, BwdWs ws,
                                                          int only_flagged) {
    using Ly = BLay<DH, DF>;
    constexpr int PF = Ly::PF, PH = Ly::PH, PW = Ly::PW, H2 = Ly::H2;
    constexpr int NC = DH / LPR, NF = DF / LPR;
    constexpr int NWE = DH * H2 / NT;  // dWf entries per thread
    extern __shared__ float sm[];
    float *sH = sm + Ly::oH, *sz = sm + Ly::oz, *sW = sm + Ly::oW, *sb = sm + Ly::ob;
    float *sphk = sm + Ly::ophk, *sv = sm + Ly::ov, *sq = sm + Ly::oq, *sphq = sm + Ly::ophq;
    float *sdp = sm + Ly::odp, *sdy = sm + Ly::ody, *sA = sm + Ly::oA, *srow = sm + Ly::orow;
    float* skt = sm + Ly::otile;  // window key tile [KB][PH]
    float* svt = skt + KB * PH;   // window value tile [KB][PH]
    float* sP = svt + KB * PH;    // ds per (row, key) [TS][KB]
    const int64_t unit = blockIdx.x, seg = blockIdx.y;
    const int64_t b = unit / p.Hkv, kv = unit % p.Hkv;
    const int64_t U = p.B * p.Hkv;
    const int64_t s0 = seg * p.seg_len, s1 = min64(p.L, s0 + p.seg_len);
    const int tid = threadIdx.x, r = tid / LPR, cs = tid % LPR;
    float* wsf = (float*)a.ws;
    if (only_flagged && ((const int*)wsf)[ws.flags + seg * U + unit] == 0) return;
    const T* W = (const T*)a.Wf + kv * DH * H2;
    for (int e = tid; e < DH * H2; e += NT) sW[(e / H2) * PW + e % H2] = ld(W + e);
    const float* rec = wsf + ws.fwd_rec + ((size_t)seg * U + unit) * p.rec_floats;
    for (int e = tid; e < DF * DH; e += NT) sH[(e / DH) * PH + e % DH] = seg > 0 ? rec[e] : 0.0f;
    if (tid < DF) sz[tid] = seg > 0 ? rec[DF * DH + tid] : 0.0f;
    float dw[NWE];
#pragma unroll
    for (int k = 0; k < NWE; ++k) dw[k] = 0.0f;
    float dts = 0.0f;  // thread hh < G: sum_i a_i delta_i of head hh
    __syncthreads();
    for (int64_t i0 = s0; i0 < s1; i0 += TS) {
        const int n = (int)min64(TS, s1 - i0);
        gates_cumsum_b<T, DF, FAST>((const T*)a.g, b, p.L, p.Hkv, kv, i0, n, sb);
        const int rlo = (int)min64(n, max64(0, p.w - i0));
        load_rows_p<T, DH>((const T*)a.k, b, p.L, p.Hkv, kv, i0 - p.w, rlo, n, sq);
        load_rows_p<T, DH>((const T*)a.v, b, p.L, p.Hkv, kv, i0 - p.w, rlo, n, sv);
        __syncthreads();
        phi_rows_p<DH, DF, FAST>(sq, sW, sphk, rlo, n);
        __syncthreads();
        if (a.kdec != nullptr) {  // masked reading: the keys enter scaled by their gate products
            simt::scale_entering_keys<DF, TS, NT, FAST>(sphk, a.kdec, b, p.L, p.Hkv, kv, i0 - p.w,
                                                        rlo, n);
            __syncthreads();
        }
        for (int hh = 0; hh < p.G; ++hh) {
            const int64_t h = kv * p.G + hh;
            load_rows_p<T, DH>((const T*)a.q, b, p.L, p.Hq, h, i0, 0, n, sq);
            load_rows_p<T, DH>((const T*)a.dy, b, p.L, p.Hq, h, i0, 0, n, sdy);
            row_stats(a, p, ws, b, h, i0, n, srow);
            __syncthreads();
            phi_rows_p<DH, DF, FAST>(sq, sW, sphq, 0, n);
            // c_it = a_i (v'_t . dy_i - delta_i), t <= i
            {
                const int i = r, t = cs;
                float val = 0.0f;
                if (t <= i && i < n && t >= rlo) {
                    float d = 0.0f;
                    for (int c = 0; c < DH; ++c) d = fmaf(sv[t * PH + c], sdy[i * PH + c], d);
                    val = srow[i] * (d - srow[TS + i]);
                }
                sA[i * (TS + 1) + t] = val;
            }
            __syncthreads();
            // dphi(q_i)_f = e^{b_if} a_i (H dy_i - z delta_i)_f + sum_t e^{b_if-b_tf} phk_tf c_it
            {
                float acc[NF];
#pragma unroll
                for (int j = 0; j < NF; ++j) acc[j] = 0.0f;
                for (int c = 0; c < DH; ++c) {
                    const float dyc = sdy[r * PH + c];
#pragma unroll
                    for (int j = 0; j < NF; ++j)
                        acc[j] = fmaf(sH[(cs + LPR * j) * PH + c], dyc, acc[j]);
                }
                const float ai = srow[r], dl = srow[TS + r];
#pragma unroll
                for (int j = 0; j < NF; ++j) {
                    const int f = cs + LPR * j;
                    const float bi = sb[r * PF + f];
                    float v = ex<FAST>(bi) * ai * (acc[j] - sz[f] * dl);
                    for (int t = 0; t <= r; ++t)
                        v = fmaf(ex<FAST>(bi - sb[t * PF + f]) * sphk[t * PF + f],
                                 sA[r * (TS + 1) + t], v);
                    sdp[r * PF + f] = r < n ? v : 0.0f;
                }
            }
            __syncthreads();
            // phi(q)-side of dB, summed over the group's heads in a fixed order
            for (int e = tid; e < TS * DF; e += NT) {
                const int t = e / DF, f = e % DF;
                if (t < n) {
                    float* dst = wsf + ws.dB + ((b * p.L + i0 + t) * p.Hkv + kv) * DF + f;
                    const float v = sphq[t * PF + f] * sdp[t * PF + f];
                    *dst = hh == 0 ? v : *dst + v;
                }
            }
            __syncthreads();
            phi_backward_rows<DF>(sphq, sdp);  // du in sdp[r][0..D/2)
            __syncthreads();
            // dWf += q^T du  (thread-owned entries, fixed order)
#pragma unroll
            for (int k = 0; k < NWE; ++k) {
                const int e = tid + NT * k, c = e / H2, f = e % H2;
                float s = 0.0f;
                for (int t = 0; t < n; ++t) s = fmaf(sq[t * PH + c], sdp[t * PF + f], s);
                dw[k] += s;
            }
            // dq_i = Wf du_i + window part
            float dq[NC];
#pragma unroll
            for (int j = 0; j < NC; ++j) {
                const int c = cs + LPR * j;
                float s = 0.0f;
                for (int f = 0; f < H2; ++f) s = fmaf(sW[c * PW + f], sdp[r * PF + f], s);
                dq[j] = s;
            }
            const float dl = srow[TS + r], lse = srow[2 * TS + r];
            const int64_t i = i0 + r;
            const int64_t jlo = max64(0, i0 - p.w + 1), jhi = i0 + n - 1;
            // (the tensor-core window kernel adds the window part afterwards when it runs)
            for (int64_t j0 = jlo; !a.win_tc && j0 <= jhi; j0 += KB) {
                __syncthreads();
                for (int e = tid; e < KB * DH; e += NT) {
                    const int t = e / DH, c = e % DH;
                    const int64_t j = j0 + t;
                    float kx = 0.0f, vx = 0.0f;
                    if (j <= jhi) {
                        kx = ld((const T*)a.k + ((b * p.L + j) * p.Hkv + kv) * DH + c);
                        vx = ld((const T*)a.v + ((b * p.L + j) * p.Hkv + kv) * DH + c);
                    }
                    skt[t * PH + c] = kx;
                    svt[t * PH + c] = vx;
                }
                __syncthreads();
                {
                    const int64_t j = j0 + cs;
                    const bool valid = (r < n) && (j <= i) && (j > i - p.w) && (j <= jhi);
                    float s = 0.0f, dv = 0.0f;
                    for (int c = 0; c < DH; ++c) {
                        s = fmaf(sq[r * PH + c], skt[cs * PH + c], s);
                        dv = fmaf(sdy[r * PH + c], svt[cs * PH + c], dv);
                    }
                    const float pij = valid ? ex<FAST>(s * p.scale - lse) : 0.0f;
                    sP[r * KB + cs] = pij * (dv - dl);
                }
                __syncwarp();
                for (int t = 0; t < KB; ++t) {
                    const float ds = sP[r * KB + t] * p.scale;
#pragma unroll
                    for (int j = 0; j < NC; ++j) dq[j] = fmaf(ds, skt[t * PH + cs + LPR * j], dq[j]);
                }
            }
            if (r < n) {
                T* dqr = (T*)a.dq + ((b * p.L + i) * p.Hq + h) * DH;
#pragma unroll
                for (int j = 0; j < NC; ++j) st(dqr + cs + LPR * j, dq[j]);
            }
            // sink statistic of this head: sum over valid rows of a_i delta_i (fixed order)
            __syncthreads();
            if (tid == hh) {
                float s = 0.0f;
                for (int t = 0; t < n; ++t) s = fmaf(srow[t], srow[TS + t], s);
                dts += s;
            }
            __syncthreads();
        }
        state_step<DH, DF, FAST>(sH, sz, sphk, sv, sb);
    }
    float* dWp = wsf + ws.dW + ((size_t)seg * U + unit) * (size_t)(DH * H2);
#pragma unroll
    for (int k = 0; k < NWE; ++k) dWp[tid + NT * k] = dw[k];
    if (tid < p.G) wsf[ws.dt + ((size_t)seg * U + unit) * p.G + tid] = dts;
}

// ---------------------------------------------------------------------------------------
// Reverse segment pass: contribution of a segment to the state adjoint at its start,
// sum_i e^{B_i - B_start} phi(q_i) g^_i^T over the segment's rows (zero adjoint at its
// end), and its total log-decay.  Record layout as the forward records: [D][d], [D], [D].
template <typename T, int DH, int DF, bool FAST>
__global__ void __launch_bounds__(NT, 1) bwd_reverse_local(Plan p, BwdArgs a, BwdWs ws) {
    using Ly = BLay<DH, DF>;
    constexpr int PF = Ly::PF, PH = Ly::PH, PW = Ly::PW, H2 = Ly::H2;
    extern __shared__ float sm[];
    float *sH = sm + Ly::oH, *sz = sm + Ly::oz, *sW = sm + Ly::oW, *sb = sm + Ly::ob;
    float *sq = sm + Ly::oq, *sphq = sm + Ly::ophq, *sdy = sm + Ly::ody, *srow = sm + Ly::orow;
    const int64_t unit = blockIdx.x, seg = blockIdx.y + 1;
    const int64_t b = unit / p.Hkv, kv = unit % p.Hkv;
    const int64_t U = p.B * p.Hkv;
    const int64_t s0 = seg * p.seg_len, s1 = min64(p.L, s0 + p.seg_len);
    const int tid = threadIdx.x;
    float* wsf = (float*)a.ws;
    const T* W = (const T*)a.Wf + kv * DH * H2;
    for (int e = tid; e < DH * H2; e += NT) sW[(e / H2) * PW + e % H2] = ld(W + e);
    for (int e = tid; e < DF * DH; e += NT) sH[(e / DH) * PH + e % DH] = 0.0f;
    if (tid < DF) sz[tid] = 0.0f;
    float lam_tot = 0.0f;
    __syncthreads();
    const int64_t nch = (s1 - s0 + TS - 1) / TS;
    for (int64_t ci = nch - 1; ci >= 0; --ci) {
        const int64_t i0 = s0 + ci * TS;
        const int n = (int)min64(TS, s1 - i0);
        gates_cumsum_b<T, DF, FAST>((const T*)a.g, b, p.L, p.Hkv, kv, i0, n, sb);
        for (int e = tid; e < DF * DH; e += NT) {
            const int f = e / DH, c = e % DH;
            sH[f * PH + c] *= ex<FAST>(sb[(TS - 1) * PF + f]);
        }
        if (tid < DF) {
            sz[tid] *= ex<FAST>(sb[(TS - 1) * PF + tid]);
            lam_tot += sb[(TS - 1) * PF + tid];
        }
        __syncthreads();
        for (int hh = 0; hh < p.G; ++hh) {
            const int64_t h = kv * p.G + hh;
            load_rows_p<T, DH>((const T*)a.q, b, p.L, p.Hq, h, i0, 0, n, sq);
            load_rows_p<T, DH>((const T*)a.dy, b, p.L, p.Hq, h, i0, 0, n, sdy);
            row_stats(a, p, ws, b, h, i0, n, srow);
            __syncthreads();
            phi_rows_p<DH, DF, FAST>(sq, sW, sphq, 0, n);
            __syncthreads();
            adjoint_add<DH, DF, FAST>(sH, sz, sphq, sdy, sb, srow, n);
        }
    }
    float* rec = wsf + ws.rev_rec + ((size_t)seg * U + unit) * p.rec_floats;
    for (int e = tid; e < DF * DH; e += NT) rec[e] = sH[(e / DH) * PH + e % DH];
    if (tid < DF) {
        rec[DF * DH + tid] = sz[tid];
        rec[DF * DH + DF + tid] = lam_tot;
    }
}

// Reverse exclusive scan, in place: record p becomes the adjoint at the end of segment p.
__global__ void bwd_reverse_scan(Plan p, float* rec0) {
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t unit = blockIdx.y;
    const int64_t nE = p.D * p.d + p.D;
    if (e >= nE) return;
    const int64_t f = e < p.D * p.d ? e / p.d : e - p.D * p.d;
    const int64_t U = p.B * p.Hkv;
    // records are read eight at a time before any is overwritten (one round trip per group)
    constexpr int KG = 8;
    float carry = 0.0f;
    for (int64_t s0 = p.P - 1; s0 >= 0; s0 -= KG) {
        float dH[KG], lam[KG];
#pragma unroll
        for (int k = 0; k < KG; ++k) {
            const int64_t sg = s0 - k;
            const float* rec = rec0 + ((size_t)(sg >= 0 ? sg : 0) * U + unit) * p.rec_floats;
            dH[k] = sg >= 1 ? rec[e] : 0.0f;
            lam[k] = sg >= 1 ? rec[p.D * p.d + p.D + f] : 0.0f;
        }
#pragma unroll
        for (int k = 0; k < KG; ++k) {
            const int64_t sg = s0 - k;
            if (sg >= 0) {
                rec0[((size_t)sg * U + unit) * p.rec_floats + e] = carry;
                carry = expf(lam[k]) * carry + dH[k];
            }
        }
    }
}

// ---------------------------------------------------------------------------------------
// Reverse-direction walk: state parts of dk, dv (keys t - w of the delayed stream),
// phi(k')-side of dB and the reverse cumulative sum of dB inside the segment, dWf partials.
// Every decay is e^{difference of cumulative log-gates} taken per pair and arranged as
// e^{non-positive}, so strongly closed gates (Lizard summary sec. 2-C: products that underflow)
// cost nothing in accuracy.
template <typename T, int DH, int DF, bool FAST>
__global__ void __launch_bounds__(NT, 1) bwd_reverse_walk(Plan p, BwdArgs a, BwdWs ws,
                                                          int only_flagged) {
    using Ly = BLay<DH, DF>;
    constexpr int PF = Ly::PF, PH = Ly::PH, PW = Ly::PW, H2 = Ly::H2;
    constexpr int NC = DH / LPR, NF = DF / LPR;
    constexpr int NWE = DH * H2 / NT;
    extern __shared__ float sm[];
    float *sH = sm + Ly::oH, *sz = sm + Ly::oz, *sW = sm + Ly::oW, *sb = sm + Ly::ob;
    float *sphk = sm + Ly::ophk, *sv = sm + Ly::ov, *sq = sm + Ly::oq, *sphq = sm + Ly::ophq;
    float *sdp = sm + Ly::odp, *sdy = sm + Ly::ody, *sA = sm + Ly::oA, *sA2 = sm + Ly::oA2;
    float* srow = sm + Ly::orow;
    const int64_t unit = blockIdx.x, seg = blockIdx.y;
    const int64_t b = unit / p.Hkv, kv = unit % p.Hkv;
    const int64_t U = p.B * p.Hkv;
    const int64_t s0 = seg * p.seg_len, s1 = min64(p.L, s0 + p.seg_len);
    const int tid = threadIdx.x, r = tid / LPR, cs = tid % LPR;
    float* wsf = (float*)a.ws;
    if (only_flagged && ((const int*)wsf)[ws.flags + seg * U + unit] == 0) return;
    const T* W = (const T*)a.Wf + kv * DH * H2;
    for (int e = tid; e < DH * H2; e += NT) sW[(e / H2) * PW + e % H2] = ld(W + e);
    const float* rec = wsf + ws.rev_rec + ((size_t)seg * U + unit) * p.rec_floats;
    const bool last = seg == p.P - 1;
    for (int e = tid; e < DF * DH; e += NT) sH[(e / DH) * PH + e % DH] = last ? 0.0f : rec[e];
    if (tid < DF) sz[tid] = last ? 0.0f : rec[DF * DH + tid];
    float dw[NWE];
#pragma unroll
    for (int k = 0; k < NWE; ++k) dw[k] = 0.0f;
    float carry = 0.0f;  // thread f < DF: sum of dB over later steps of this segment
    __syncthreads();
    const int64_t nch = (s1 - s0 + TS - 1) / TS;
    for (int64_t ci = nch - 1; ci >= 0; --ci) {
        const int64_t i0 = s0 + ci * TS;
        const int n = (int)min64(TS, s1 - i0);
        gates_cumsum_b<T, DF, FAST>((const T*)a.g, b, p.L, p.Hkv, kv, i0, n, sb);
        const int rlo = (int)min64(n, max64(0, p.w - i0));
        load_rows_p<T, DH>((const T*)a.k, b, p.L, p.Hkv, kv, i0 - p.w, rlo, n, sq);
        load_rows_p<T, DH>((const T*)a.v, b, p.L, p.Hkv, kv, i0 - p.w, rlo, n, sv);
        __syncthreads();
        phi_rows_p<DH, DF, FAST>(sq, sW, sphk, rlo, n);
        __syncthreads();
        if (a.kdec != nullptr) {  // masked reading: sphk holds c (.) phi(k'), the entering value
            simt::scale_entering_keys<DF, TS, NT, FAST>(sphk, a.kdec, b, p.L, p.Hkv, kv, i0 - p.w,
                                                        rlo, n);
            __syncthreads();
        }
        // terms through the step's end: dphk_t = e^{bl - b_t} (.) (dH v'_t + dz),
        // dv'_t = sum_f e^{bl_f - b_tf} phk_tf dH[f][.]   (row t = r, in registers)
        float dk_acc[NF], dv_acc[NC];
        {
#pragma unroll
            for (int j = 0; j < NF; ++j) dk_acc[j] = 0.0f;
            for (int c = 0; c < DH; ++c) {
                const float vc = sv[r * PH + c];
#pragma unroll
                for (int j = 0; j < NF; ++j) dk_acc[j] = fmaf(sH[(cs + LPR * j) * PH + c], vc, dk_acc[j]);
            }
#pragma unroll
            for (int j = 0; j < NF; ++j) {
                const int f = cs + LPR * j;
                dk_acc[j] = ex<FAST>(sb[(TS - 1) * PF + f] - sb[r * PF + f]) * (dk_acc[j] + sz[f]);
            }
            // weights e^{bl - b_t} phk_t of the end term, once per (row, feature) (sdp is free)
            for (int e = tid; e < TS * DF; e += NT) {
                const int t = e / DF, f = e % DF;
                sdp[t * PF + f] = ex<FAST>(sb[(TS - 1) * PF + f] - sb[t * PF + f]) * sphk[t * PF + f];
            }
            __syncthreads();
#pragma unroll
            for (int j = 0; j < NC; ++j) dv_acc[j] = 0.0f;
            for (int f = 0; f < DF; ++f) {
                const float w_ = sdp[r * PF + f];
#pragma unroll
                for (int j = 0; j < NC; ++j) dv_acc[j] = fmaf(sH[f * PH + cs + LPR * j], w_, dv_acc[j]);
            }
        }
        __syncthreads();
        // the adjoint decays back over the step; the step's own rows are added per head
        for (int e = tid; e < DF * DH; e += NT) {
            const int f = e / DH, c = e % DH;
            sH[f * PH + c] *= ex<FAST>(sb[(TS - 1) * PF + f]);
        }
        if (tid < DF) sz[tid] *= ex<FAST>(sb[(TS - 1) * PF + tid]);
        __syncthreads();
        for (int hh = 0; hh < p.G; ++hh) {
            const int64_t h = kv * p.G + hh;
            load_rows_p<T, DH>((const T*)a.q, b, p.L, p.Hq, h, i0, 0, n, sq);
            load_rows_p<T, DH>((const T*)a.dy, b, p.L, p.Hq, h, i0, 0, n, sdy);
            row_stats(a, p, ws, b, h, i0, n, srow);
            __syncthreads();
            phi_rows_p<DH, DF, FAST>(sq, sW, sphq, 0, n);
            __syncthreads();
            // c_it = a_i (v'_t.dy_i - delta_i); A_it a_i = a_i sum_f phq_if phk_tf e^{b_if - b_tf}
            {
                const int i = r, t = cs;
                float cv = 0.0f, av = 0.0f;
                if (t <= i && i < n && t >= rlo) {
                    float d = 0.0f;
                    for (int c = 0; c < DH; ++c) d = fmaf(sv[t * PH + c], sdy[i * PH + c], d);
                    cv = srow[i] * (d - srow[TS + i]);
                    float s = 0.0f;
                    for (int f = 0; f < DF; ++f)
                        s = fmaf(sphq[i * PF + f] * sphk[t * PF + f],
                                 ex<FAST>(sb[i * PF + f] - sb[t * PF + f]), s);
                    av = s * srow[i];
                }
                sA[i * (TS + 1) + t] = cv;
                sA2[i * (TS + 1) + t] = av;
            }
            __syncthreads();
            // intra terms for row t = r: dphk += sum_{i>=t} e^{b_i-b_t} phq_i c_it; dv' += sum_i A a dy_i
#pragma unroll
            for (int j = 0; j < NF; ++j) {
                const int f = cs + LPR * j;
                const float bt = sb[r * PF + f];
                float v = 0.0f;
                for (int i = r; i < n; ++i)
                    v = fmaf(sphq[i * PF + f] * ex<FAST>(sb[i * PF + f] - bt), sA[i * (TS + 1) + r], v);
                dk_acc[j] += v;
            }
#pragma unroll
            for (int j = 0; j < NC; ++j) {
                const int c = cs + LPR * j;
                float v = 0.0f;
                for (int i = r; i < n; ++i) v = fmaf(sA2[i * (TS + 1) + r], sdy[i * PH + c], v);
                dv_acc[j] += v;
            }
            __syncthreads();
            adjoint_add<DH, DF, FAST>(sH, sz, sphq, sdy, sb, srow, n);
        }
        // dphk into sdp (rows outside [rlo, n) are zero)
#pragma unroll
        for (int j = 0; j < NF; ++j)
            sdp[r * PF + cs + LPR * j] = (r >= rlo && r < n) ? dk_acc[j] : 0.0f;
        __syncthreads();
        // dB = (phi(q)-side, from the forward walk) - phk (.) dphk; reverse cumsum in place.
        // Masked reading: the key's term belongs to its own row t - w (its factor
        // e^{-b} is taken at the key's position), so it goes to the separate array kkey, and
        // phi's backward takes the unscaled map with dphi = c (.) dphi(c phi).
        if (tid < DF) {
            const int f = tid;
            for (int t = n - 1; t >= 0; --t) {
                float* src = wsf + ws.dB + ((b * p.L + i0 + t) * p.Hkv + kv) * DF + f;
                carry += a.kkey != nullptr ? *src : *src - sphk[t * PF + f] * sdp[t * PF + f];
                *src = carry;
            }
        }
        if (a.kkey != nullptr) {
            for (int e = tid; e < TS * DF; e += NT) {
                const int t = e / DF, f = e % DF;
                if (t >= rlo && t < n)
                    a.kkey[((b * p.L + i0 + t - p.w) * p.Hkv + kv) * DF + f] =
                        sphk[t * PF + f] * sdp[t * PF + f];
            }
            __syncthreads();
            load_rows_p<T, DH>((const T*)a.k, b, p.L, p.Hkv, kv, i0 - p.w, rlo, n, sq);
            __syncthreads();
            phi_rows_p<DH, DF, FAST>(sq, sW, sphk, rlo, n);
            for (int e = tid; e < TS * DF; e += NT) {
                const int t = e / DF, f = e % DF;
                if (t >= rlo && t < n)
                    sdp[t * PF + f] *= ex<FAST>(a.kdec[((b * p.L + i0 + t - p.w) * p.Hkv + kv) * DF + f]);
            }
        }
        __syncthreads();
        phi_backward_rows<DF>(sphk, sdp);  // du of the delayed keys
        // raw k' rows again (sq holds q now)
        load_rows_p<T, DH>((const T*)a.k, b, p.L, p.Hkv, kv, i0 - p.w, rlo, n, sq);
        __syncthreads();
#pragma unroll
        for (int k = 0; k < NWE; ++k) {
            const int e = tid + NT * k, c = e / H2, f = e % H2;
            float s = 0.0f;
            for (int t = rlo; t < n; ++t) s = fmaf(sq[t * PH + c], sdp[t * PF + f], s);
            dw[k] += s;
        }
        if (r >= rlo && r < n) {
            const int64_t j = i0 + r - p.w;
            T* dkr = (T*)a.dk + ((b * p.L + j) * p.Hkv + kv) * DH;
            T* dvr = (T*)a.dv + ((b * p.L + j) * p.Hkv + kv) * DH;
#pragma unroll
            for (int jj = 0; jj < NC; ++jj) {
                const int c = cs + LPR * jj;
                float s = 0.0f;
                for (int f = 0; f < H2; ++f) s = fmaf(sW[c * PW + f], sdp[r * PF + f], s);
                st(dkr + c, s);
                st(dvr + c, dv_acc[jj]);
            }
        }
        __syncthreads();
    }
    float* dWp = wsf + ws.dW + ((size_t)(p.Pmax + seg) * U + unit) * (size_t)(DH * H2);
#pragma unroll
    for (int k = 0; k < NWE; ++k) dWp[tid + NT * k] = dw[k];
    if (tid < DF) wsf[ws.tot + ((size_t)seg * U + unit) * DF + tid] = carry;
}

// Segments whose gates close too hard for the tensor-core walks' factored decays: flag
// (segment, unit) when some feature's cumulative log-gate falls by more than 60 over one of
// the 16-token halves of the walks' 32-token steps (Lizard summary sec. 2-C: products of such
// gates underflow).  128 threads: 16 per token row (8 features each) times 8 halves at a
// time, so four CTAs fit an SM beside each other and one wave holds the grid.
constexpr int kFlagThreads = 128;
__global__ void __launch_bounds__(kFlagThreads) bwd_gate_flags(Plan p, const __nv_bfloat16* g,
                                                               int* flags) {
    const int64_t unit = blockIdx.x, seg = blockIdx.y;
    const int64_t b = unit / p.Hkv, kv = unit % p.Hkv;
    const int64_t s0 = seg * p.seg_len, s1 = min64(p.L, s0 + p.seg_len);
    // thread: features 8 c8 .. + 7 of the 16-token halves s0 + 16 hq, + 128, ...: one 16-byte
    // load per token, the half's 16 loads in flight together.  A half's log-decay is
    // sum_t log sigmoid(g_t) = sum_t min(g_t, 0) - ln prod_t (1 + e^{-|g_t|}); every factor of
    // the product lies in (1, 2], so 16 of them stay finite and one logarithm per half does
    // (fast exponentials and logarithm: the threshold decides between two exact walks)
    const int c8 = threadIdx.x & 15, hq = threadIdx.x >> 4;
    const int64_t stride = p.Hkv * 128;
    bool closed = false;
    for (int64_t h0 = s0 + 16 * hq; h0 < s1; h0 += 16 * (kFlagThreads / 16)) {
        const int nt = (int)min64(16, s1 - h0);
        const __nv_bfloat16* row = g + ((b * p.L + h0) * p.Hkv + kv) * 128 + 8 * c8;
        uint4 v[16];
#pragma unroll
        for (int t = 0; t < 16; ++t)
            v[t] = t < nt ? *reinterpret_cast<const uint4*>(row + t * stride) : make_uint4(0u, 0u, 0u, 0u);
        float lo[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        float pr[8] = {1.0f, 1.0f, 1.0f, 1.0f, 1.0f, 1.0f, 1.0f, 1.0f};
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            if (t >= nt) break;
            const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&v[t]);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float x = __bfloat162float(e[k]);
                lo[k] += fminf(x, 0.0f);
                pr[k] *= 1.0f + __expf(-fabsf(x));
            }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) closed |= !(lo[k] - __logf(pr[k]) >= -60.0f);
    }
    const int any = __syncthreads_or(closed);
    if (threadIdx.x == 0) flags[seg * p.B * p.Hkv + unit] = any ? 1 : 0;
}
// ---------------------------------------------------------------------------------------
// Window part of dk, dv, key-centric: keys j of a 32-key tile, queries i in [j, j + w).
// Keys with j + w < L already hold their state parts; the window part is added to them.
template <typename T, int DH, bool FAST>
__global__ void __launch_bounds__(NT) bwd_window_keys(Plan p, BwdArgs a, BwdWs ws) {
    constexpr int PH = DH + 1, QT = 8;  // query tokens per tile
    extern __shared__ float sm[];
    float* sk = sm;                  // [32][PH]
    float* sv = sk + 32 * PH;        // [32][PH]
    float* sq = sv + 32 * PH;        // [QT*G][PH]
    float* sdy = sq + QT * 8 * PH;   // [QT*G][PH]
    float* srow = sdy + QT * 8 * PH; // lse, delta [2][QT*G]
    float* sP = srow + 2 * QT * 8;   // p [QT*G][33]
    float* sD = sP + QT * 8 * 33;    // ds [QT*G][33]
    const int64_t unit = blockIdx.y, j0 = (int64_t)blockIdx.x * 32;
    const int64_t b = unit / p.Hkv, kv = unit % p.Hkv;
    const int G = (int)p.G, RQ = QT * G;
    const int tid = threadIdx.x;
    for (int e = tid; e < 32 * DH; e += NT) {
        const int t = e / DH, c = e % DH;
        const int64_t j = j0 + t;
        sk[t * PH + c] = j < p.L ? ld((const T*)a.k + ((b * p.L + j) * p.Hkv + kv) * DH + c) : 0.0f;
        sv[t * PH + c] = j < p.L ? ld((const T*)a.v + ((b * p.L + j) * p.Hkv + kv) * DH + c) : 0.0f;
    }
    // accumulators: thread owns (key kk, columns c = cc + 8 m) for dk and dv
    const int kk = tid >> 3, cc = tid & 7;
    float ak[DH / 8], av[DH / 8];
#pragma unroll
    for (int m = 0; m < DH / 8; ++m) ak[m] = av[m] = 0.0f;
    const int64_t ihi = min64(p.L, j0 + 32 + p.w - 1);
    for (int64_t q0 = j0; q0 < ihi; q0 += QT) {
        __syncthreads();
        for (int e = tid; e < RQ * DH; e += NT) {
            const int rr = e / DH, c = e % DH, t = rr / G, hh = rr % G;
            const int64_t i = q0 + t;
            float qx = 0.0f, dx = 0.0f;
            if (i < ihi) {
                const int64_t off = ((b * p.L + i) * p.Hq + kv * G + hh) * DH + c;
                qx = ld((const T*)a.q + off);
                dx = ld((const T*)a.dy + off);
            }
            sq[rr * PH + c] = qx;
            sdy[rr * PH + c] = dx;
        }
        for (int rr = tid; rr < RQ; rr += NT) {
            const int t = rr / G, hh = rr % G;
            const int64_t i = q0 + t;
            float lse = 0.0f, dl = 0.0f;
            if (i < ihi) {
                const int64_t off = ((b * p.L + i) * p.Hq + kv * G + hh);
                lse = a.lse[off];
                dl = ((const float*)a.ws)[ws.rows + p.B * p.L * p.Hq + off];
            }
            srow[rr] = lse;
            srow[RQ + rr] = dl;
        }
        __syncthreads();
        for (int e = tid; e < RQ * 32; e += NT) {
            const int rr = e / 32, t = e % 32, tq = rr / G;
            const int64_t i = q0 + tq, j = j0 + t;
            float pv = 0.0f, dsv = 0.0f;
            if (i < ihi && j < p.L && j <= i && i < j + p.w) {
                float s = 0.0f, dv = 0.0f;
                for (int c = 0; c < DH; ++c) {
                    s = fmaf(sq[rr * PH + c], sk[t * PH + c], s);
                    dv = fmaf(sdy[rr * PH + c], sv[t * PH + c], dv);
                }
                pv = ex<FAST>(s * p.scale - srow[rr]);
                dsv = pv * (dv - srow[RQ + rr]) * p.scale;
            }
            sP[rr * 33 + t] = pv;
            sD[rr * 33 + t] = dsv;
        }
        __syncthreads();
        for (int rr = 0; rr < RQ; ++rr) {
            const float pv = sP[rr * 33 + kk], dsv = sD[rr * 33 + kk];
#pragma unroll
            for (int m = 0; m < DH / 8; ++m) {
                ak[m] = fmaf(dsv, sq[rr * PH + cc + 8 * m], ak[m]);
                av[m] = fmaf(pv, sdy[rr * PH + cc + 8 * m], av[m]);
            }
        }
    }
    const int64_t j = j0 + kk;
    if (j < p.L) {
        const bool has_state = j + p.w < p.L;
        T* dkr = (T*)a.dk + ((b * p.L + j) * p.Hkv + kv) * DH;
        T* dvr = (T*)a.dv + ((b * p.L + j) * p.Hkv + kv) * DH;
#pragma unroll
        for (int m = 0; m < DH / 8; ++m) {
            const int c = cc + 8 * m;
            st(dkr + c, ak[m] + (has_state ? ld(dkr + c) : 0.0f));
            st(dvr + c, av[m] + (has_state ? ld(dvr + c) : 0.0f));
        }
    }
}

// dg = (sum_{s >= u} dB_s) (1 - sigmoid(g_u)); the in-segment sums are in the scratch,
// later segments add their totals.  Decay readings: the lagged one ran every kernel on the
// gates moved w tokens later, so gate j takes the adjoint of moved row j + w (and the gates
// of the last w tokens, never used, get 0); the masked one subtracts the suffix sums of the
// key-side terms kept at the keys' own rows.
template <typename T>
__global__ void bwd_gates(Plan p, BwdArgs a, BwdWs ws) {
    // eight consecutive features of one (batch, token, KV head) row per thread
    const int64_t total8 = p.B * p.L * p.Hkv * p.D / 8;
    const int64_t e8 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e8 >= total8) return;
    const int64_t e = e8 * 8;
    const int64_t rowj = e / p.D;                   // (b L + j) Hkv + kv: the gate written
    const int f0 = (int)(e - rowj * p.D);
    const int64_t kv = rowj % p.Hkv, bj = rowj / p.Hkv;
    const int64_t j = bj % p.L, b = bj / p.L;
    const int64_t i = j + a.glag;                   // the row of the adjoint it takes
    if (i >= p.L) {
        if constexpr (sizeof(T) == 2)
            *reinterpret_cast<uint4*>((__nv_bfloat16*)a.dg + e) = make_uint4(0u, 0u, 0u, 0u);
        else
#pragma unroll
            for (int k = 0; k < 8; ++k) st((T*)a.dg + e + k, 0.0f);
        return;
    }
    const int64_t ei = e + a.glag * p.Hkv * p.D;
    const int64_t seg = i / p.seg_len;
    const int64_t U = p.B * p.Hkv, unit = b * p.Hkv + kv;
    const float* wsf = (const float*)a.ws;
    // tot holds, per segment, the sum of dB over all later segments (bwd_tot_suffix)
    const float* tot = wsf + ws.tot + ((size_t)seg * U + unit) * p.D + f0;
    const float4 d0 = *reinterpret_cast<const float4*>(wsf + ws.dB + ei);
    const float4 d1 = *reinterpret_cast<const float4*>(wsf + ws.dB + ei + 4);
    const float4 t0 = *reinterpret_cast<const float4*>(tot);
    const float4 t1 = *reinterpret_cast<const float4*>(tot + 4);
    float dv[8] = {d0.x + t0.x, d0.y + t0.y, d0.z + t0.z, d0.w + t0.w,
                   d1.x + t1.x, d1.y + t1.y, d1.z + t1.z, d1.w + t1.w};
    if (a.kkey != nullptr) {
        const float4 k0 = *reinterpret_cast<const float4*>(a.kkey + e);
        const float4 k1 = *reinterpret_cast<const float4*>(a.kkey + e + 4);
        const float kv8[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) dv[k] -= kv8[k];
    }
    if constexpr (sizeof(T) == 2) {
        // d log sigmoid(g)/dg = 1 - sigmoid(g) = 1 / (1 + e^g), which keeps its relative
        // precision for large g; eight gates in one 16-byte load
        const uint4 gw = *reinterpret_cast<const uint4*>((const __nv_bfloat16*)a.g + ei);
        const uint32_t w[4] = {gw.x, gw.y, gw.z, gw.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float g0 = __uint_as_float(w[k] << 16), g1 = __uint_as_float(w[k] & 0xFFFF0000u);
            const __nv_bfloat162 h =
                __floats2bfloat162_rn(dv[2 * k] / (1.0f + expf(g0)), dv[2 * k + 1] / (1.0f + expf(g1)));
            o[k] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>((__nv_bfloat16*)a.dg + e) = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            st((T*)a.dg + e + k, dv[k] / (1.0f + expf(ld((const T*)a.g + ei + k))));
    }
}

// Segment totals of dB -> exclusive suffix sums over the segments (later segments first).
__global__ void bwd_tot_suffix(Plan p, float* tot) {
    const int64_t U = p.B * p.Hkv;
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // unit * D + f
    if (e >= U * p.D) return;
    // totals read eight at a time before any is overwritten (one round trip per group
    // instead of one per segment)
    constexpr int KG = 8;
    float run = 0.0f;
    for (int64_t s0 = p.P - 1; s0 >= 0; s0 -= KG) {
        float t[KG];
#pragma unroll
        for (int k = 0; k < KG; ++k) t[k] = s0 - k >= 0 ? tot[(size_t)(s0 - k) * U * p.D + e] : 0.0f;
#pragma unroll
        for (int k = 0; k < KG; ++k) {
            if (s0 - k >= 0) {
                tot[(size_t)(s0 - k) * U * p.D + e] = run;
                run += t[k];
            }
        }
    }
}

// dWf[kv] = sum over batch, segments and both walks (fixed order); dsinks likewise.  Each
// dWf entry takes four threads, thread `part` summing the segments sg = part mod 4 of both
// walks (so four times as many loads are in flight), added in a fixed order.
constexpr int kRedCols = 64, kRedParts = 4;

__global__ void __launch_bounds__(kRedCols * kRedParts) bwd_reduce(Plan p, BwdArgs a, BwdWs ws) {
    __shared__ float part_sum[kRedParts][kRedCols];
    const int64_t nW = p.d * (p.D / 2);
    const int col = threadIdx.x % kRedCols, part = threadIdx.x / kRedCols;
    const int64_t e = (int64_t)blockIdx.x * kRedCols + col;
    const float* wsf = (const float*)a.ws;
    const int64_t U = p.B * p.Hkv;
    const bool has = e < p.Hkv * nW;
    float sum = 0.0f;
    if (has) {
        const int64_t kv = e / nW, x = e % nW;
        const size_t bs = (size_t)p.Hkv * (size_t)nW;
        for (int w2 = 0; w2 < 2; ++w2)
            for (int64_t sg = part; sg < p.P; sg += kRedParts) {
                const float* src = wsf + ws.dW + ((size_t)(w2 * p.Pmax + sg) * U + kv) * nW + x;
                for (int64_t b = 0; b < p.B; ++b) sum += src[b * bs];
            }
    }
    part_sum[part][col] = sum;
    __syncthreads();
    if (has && part == 0)
        a.dWf[e] = (part_sum[0][col] + part_sum[1][col]) + (part_sum[2][col] + part_sum[3][col]);
    const int64_t et = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (et < p.Hq * p.M && a.dsinks != nullptr) {
        const int64_t h = et / p.M, kv = h / p.G, hh = h % p.G;
        float s = 0.0f;
        for (int64_t sg = 0; sg < p.P; ++sg)
            for (int64_t b = 0; b < p.B; ++b)
                s += wsf[ws.dt + ((size_t)sg * U + b * p.Hkv + kv) * p.G + hh];
        a.dsinks[et] = -expf(a.sinks[et]) * s;
    }
}

template <typename T, int DH, int DF, bool FAST>
cudaError_t bwd_impl(const Plan& p, const BwdArgs& a_in, cudaStream_t s) {
    using Ly = BLay<DH, DF>;
    const BwdWs ws = bwd_layout(p);
    BwdArgs a = a_in;
    const size_t smem = Ly::bytes;
    cudaError_t e;
    e = cudaFuncSetAttribute(bwd_forward_walk<T, DH, DF, FAST>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(bwd_reverse_local<T, DH, DF, FAST>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(bwd_reverse_walk<T, DH, DF, FAST>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const size_t wsmem = sizeof(float) * (size_t)(2 * 32 * (DH + 1) + 2 * 64 * (DH + 1) + 2 * 64 +
                                                  2 * 64 * 33);
    e = cudaFuncSetAttribute(bwd_window_keys<T, DH, FAST>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wsmem);
    if (e != cudaSuccess) return e;
    const unsigned U = (unsigned)(p.B * p.Hkv);
    float* wsf = (float*)a.ws;
    // decay readings: every kernel below reads the moved gates (LAGGED), or the SIMT walks
    // scale the entering keys and keep their gate terms apart (MASKED)
    if (p.decay == LIZARD_DECAY_LAGGED) {
        e = launch_gate_lag(p, a.g, wsf + ws.gl, s);
        if (e != cudaSuccess) return e;
        a.g = wsf + ws.gl;
        a.glag = p.w;
    } else if (p.decay == LIZARD_DECAY_MASKED) {
        e = launch_key_decay(p, a.g, wsf + ws.kd, s);
        if (e != cudaSuccess) return e;
        a.kdec = wsf + ws.kd;
        a.kkey = wsf + ws.kk;
    }
    // 0. per-row a = e^{-lse} and delta = dy . y
    {
        const int64_t nrow = p.B * p.L * p.Hq;
        if constexpr (sizeof(T) == 2 && DH == 128)
            bwd_row_table_bf16<<<(unsigned)((nrow + 8 * kRowsPerWarp - 1) / (8 * kRowsPerWarp)), 256, 0, s>>>(p, a, ws);
        else
            bwd_row_table<T, DH><<<(unsigned)((nrow + 7) / 8), 256, 0, s>>>(p, a, ws);
    }
    // 1. forward segment states (segment pass + scan) into the first record region
    if (p.P > 1) {
        FwdArgs fa{};
        fa.q = a.q;
        fa.k = a.k;
        fa.v = a.v;
        fa.g = a.g;
        fa.Wf = a.Wf;
        fa.sinks = a.sinks;
        fa.seg = wsf + ws.fwd_rec;
        fa.header = a.ws;
        fa.kdec = a.kdec;
        e = fwd_tc_supported(p) ? launch_fwd_states_tc(p, fa, s) : launch_fwd_states(p, fa, s);
        if (e != cudaSuccess) return e;
    }
    // 2. forward-direction walk.  The tensor-core walks leave the segments whose gates close
    //    too hard for their factored decays to the exact SIMT walks (flags from one pass over g)
    const bool tc_walks = a.win_tc && bwd_rev_local_tc_supported(p);
    int* flags = (int*)(wsf + ws.flags);
    if (tc_walks) {
        if constexpr (sizeof(T) == 2 && DF == 128)
            bwd_gate_flags<<<dim3(U, (unsigned)p.P), kFlagThreads, 0, s>>>(
                p, (const __nv_bfloat16*)a.g, flags);
    }
    if (a.ev_before) cudaEventRecord(a.ev_before, s);
    if (tc_walks) {
        e = launch_bwd_fwalk_tc(p, a, wsf, ws.rows, ws.fwd_rec, ws.dB, ws.dW, ws.dt, flags, s);
        if (e != cudaSuccess) return e;
    }
    bwd_forward_walk<T, DH, DF, FAST><<<dim3(U, (unsigned)p.P), NT, smem, s>>>(p, a, ws, tc_walks ? 1 : 0);
    if (a.ev_after) cudaEventRecord(a.ev_after, s);
    // window part of dq on the tensor cores (the walk above wrote the state part)
    if (a.win_tc) {
        e = launch_bwd_win_tc(p, a, wsf + ws.rows, false, s);
        if (e != cudaSuccess) return e;
    }
    // 3. reverse segment pass and scan
    if (p.P > 1) {
        if (tc_walks) {
            e = launch_bwd_rev_local_tc(p, a, wsf + ws.rows, wsf + ws.rev_rec, s);
            if (e != cudaSuccess) return e;
        } else {
            bwd_reverse_local<T, DH, DF, FAST><<<dim3(U, (unsigned)(p.P - 1)), NT, smem, s>>>(p, a, ws);
        }
        const unsigned nE = (unsigned)(p.D * p.d + p.D);
        bwd_reverse_scan<<<dim3((nE + 255) / 256, U), 256, 0, s>>>(p, wsf + ws.rev_rec);
    }
    // 4. reverse-direction walk
    if (tc_walks) {
        e = launch_bwd_rwalk_tc(p, a, wsf, ws.rows, ws.rev_rec, ws.dB, ws.dW, ws.tot, flags, s);
        if (e != cudaSuccess) return e;
    }
    bwd_reverse_walk<T, DH, DF, FAST><<<dim3(U, (unsigned)p.P), NT, smem, s>>>(p, a, ws, tc_walks ? 1 : 0);
    // 5. window parts of dk, dv
    if (a.win_tc) {
        e = launch_bwd_win_tc(p, a, wsf + ws.rows, true, s);
        if (e != cudaSuccess) return e;
    } else {
        bwd_window_keys<T, DH, FAST><<<dim3((unsigned)((p.L + 31) / 32), U), NT, wsmem, s>>>(p, a, ws);
    }
    // 6. dg, then the reductions
    const int64_t ng = p.B * p.L * p.Hkv * p.D;
    if (a.kkey != nullptr) {
        e = launch_key_suffix(p, a.kkey, wsf + ws.kt, s);
        if (e != cudaSuccess) return e;
    }
    bwd_tot_suffix<<<(unsigned)((U * p.D + 255) / 256), 256, 0, s>>>(p, wsf + ws.tot);
    bwd_gates<T><<<(unsigned)((ng / 8 + 255) / 256), 256, 0, s>>>(p, a, ws);
    // dWf: kRedCols entries per block; dsinks: one entry per thread of the same blocks
    const int64_t nW = p.d * (p.D / 2);
    const int64_t nb = max64((p.Hkv * nW + kRedCols - 1) / kRedCols,
                             (p.Hq * p.M + kRedCols * kRedParts - 1) / (kRedCols * kRedParts));
    bwd_reduce<<<(unsigned)nb, kRedCols * kRedParts, 0, s>>>(p, a, ws);
    return cudaGetLastError();
}

template <typename T, bool FAST>
cudaError_t bwd_dims(const Plan& p, const BwdArgs& a, cudaStream_t s) {
    if (p.d == 128 && p.D == 128) return bwd_impl<T, 128, 128, FAST>(p, a, s);
    if (p.d == 128 && p.D == 64) return bwd_impl<T, 128, 64, FAST>(p, a, s);
    if (p.d == 64 && p.D == 128) return bwd_impl<T, 64, 128, FAST>(p, a, s);
    if (p.d == 64 && p.D == 64) return bwd_impl<T, 64, 64, FAST>(p, a, s);
    return cudaErrorInvalidValue;
}

}  // namespace

size_t bwd_workspace_bytes(const Plan& p) { return bwd_layout(p).total; }

cudaError_t launch_bwd(const Plan& p, const BwdArgs& a, cudaStream_t s) {
    if (p.G > 8) return cudaErrorInvalidValue;
    // the walks run one CTA per (unit, segment), one CTA per SM: cut the segments so the
    // last wave is as full as the others
    Plan q = p;
    plan_segments_waves(&q, 152);
    BwdArgs b = a;
    b.win_tc = bwd_win_tc_supported(q) ? 1 : 0;
    if (q.dtype == LIZARD_F32) return bwd_dims<float, false>(q, b, s);
    return bwd_dims<__nv_bfloat16, true>(q, b, s);
}

}  // namespace lz
