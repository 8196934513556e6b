// SIMT forward of the Lizard token mixer (fp32 path, and every shape the tensor-core
// path does not cover).
//
// Lizard summary (gist.science/ko/paper/2507.09025): sec. 2-A-1 gated linear
// attention over the tokens that have left the window, sec. 2-A-2 sliding-window
// softmax with meta-memory scalars in the denominator, sec. 2-C Hedgehog feature
// map and gates in log space.  Decays are exp of differences of cumulative
// log-gates, always arranged as exp(non-positive), so nothing overflows.
//
// Three launches:
//   1. seglocal: every segment but the last computes its own state contribution
//      dH = sum_t e^{B_end - B_t} phi(k_{t-w}) v_{t-w}^T (and dz) and its total
//      log-decay dLam, starting from a zero state;
//   2. scan: an fp32 scan over segments turns those into each segment's
//      starting state H_p = e^{dLam_{p-1}} H_{p-1} + dH_{p-1};
//   3. main: one CTA per (query head, segment) walks its segment 32 tokens at a
//      time: state readout, intra-sub-chunk state term, window softmax with
//      sinks, shared-normaliser epilogue, state update.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "simt.cuh"

namespace lz {
namespace {

using namespace simt;

template <typename T, int DH, int DF, bool FAST>
__global__ void __launch_bounds__(NT, 1) fwd_simt_seglocal(Plan p, FwdArgs a) {
    using Ly = Lay<DH, DF>;
    extern __shared__ float sm[];
    float *sH = sm + Ly::oH, *sz = sm + Ly::oz, *sW = sm + Ly::oW, *sb = sm + Ly::ob;
    float *sphk = sm + Ly::ophk, *sv = sm + Ly::ov, *sq = sm + Ly::oq;
    const int64_t unit = blockIdx.x, seg = blockIdx.y;
    const int64_t b = unit / p.Hkv, kv = unit % p.Hkv;
    const int64_t s0 = seg * p.seg_len, s1 = min64(p.L, s0 + p.seg_len);
    const T* W = (const T*)a.Wf + kv * DH * (DF / 2);
    for (int e = threadIdx.x; e < DH * (DF / 2); e += NT) sW[e] = ld(W + e);
    for (int e = threadIdx.x; e < DF * DH; e += NT) sH[e] = 0.0f;
    if (threadIdx.x < DF) sz[threadIdx.x] = 0.0f;
    float lam_tot = 0.0f;  // thread f < DF: total log-decay of the segment
    __syncthreads();
    for (int64_t i0 = s0; i0 < s1; i0 += TS) {
        const int n = (int)min64(TS, s1 - i0);
        gates_cumsum<T, DF, FAST>((const T*)a.g, b, p.L, p.Hkv, kv, i0, n, sb);
        const int rlo = (int)min64(n, max64(0, p.w - i0));
        load_rows<T, DH>((const T*)a.k, b, p.L, p.Hkv, kv, i0 - p.w, rlo, n, sq, Ly::PH);
        load_rows<T, DH>((const T*)a.v, b, p.L, p.Hkv, kv, i0 - p.w, rlo, n, sv, DH);
        __syncthreads();
        phi_rows<DH, DF, FAST>(sq, sW, sphk, rlo, n);
        if (threadIdx.x < DF) lam_tot += sb[(TS - 1) * Ly::PF + threadIdx.x];
        __syncthreads();
        if (a.kdec != nullptr) {  // masked reading
            scale_entering_keys<DF, TS, NT, FAST>(sphk, a.kdec, b, p.L, p.Hkv, kv, i0 - p.w, rlo, n);
            __syncthreads();
        }
        state_update<DH, DF, FAST>(sH, sz, sphk, sv, sb);
    }
    float* rec = a.seg + ((size_t)seg * (size_t)(p.B * p.Hkv) + (size_t)unit) * p.rec_floats;
    for (int e = threadIdx.x; e < DF * DH; e += NT) rec[e] = sH[e];
    if (threadIdx.x < DF) {
        rec[DF * DH + threadIdx.x] = sz[threadIdx.x];
        rec[DF * DH + DF + threadIdx.x] = lam_tot;
    }
}

// Exclusive scan over segments, in place: record p becomes the state before segment p.
__global__ void fwd_seg_scan(Plan p, float* seg) {
    grid_dep_wait();  // the segment records of the pass before
    grid_dep_launch();
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t unit = blockIdx.y;
    const int64_t nE = p.D * p.d + p.D;
    if (e >= nE) return;
    const int64_t f = e < p.D * p.d ? e / p.d : e - p.D * p.d;
    const int64_t U = p.B * p.Hkv;
    // records are read eight at a time before any is overwritten, so the loads of a group
    // are in flight together instead of one memory round trip per segment
    constexpr int KG = 8;
    float carry = 0.0f;
    for (int64_t s0 = 0; s0 < p.P; s0 += KG) {
        float dH[KG], lam[KG];
#pragma unroll
        for (int k = 0; k < KG; ++k) {
            const int64_t s = s0 + k;
            const float* rec = seg + ((size_t)s * U + unit) * p.rec_floats;
            dH[k] = s < p.P - 1 ? rec[e] : 0.0f;
            lam[k] = s < p.P - 1 ? rec[p.D * p.d + p.D + f] : 0.0f;
        }
#pragma unroll
        for (int k = 0; k < KG; ++k) {
            const int64_t s = s0 + k;
            if (s < p.P) {
                seg[((size_t)s * U + unit) * p.rec_floats + e] = carry;
                carry = expf(lam[k]) * carry + dH[k];
            }
        }
    }
}

// One query head h of batch entry b over tokens [s0, s1), starting from the state in `rec`
// ([D][d] then [D]; null: the zero state).  s0 is a multiple of the 32-token step.
template <typename T, int DH, int DF, bool FAST>
__device__ __forceinline__ void walk_head(const Plan& p, const FwdArgs& a, int64_t b, int64_t h,
                                          int64_t s0, int64_t s1, const float* rec, float* sm) {
    using Ly = Lay<DH, DF>;
    constexpr int PF = Ly::PF, PH = Ly::PH, NC = DH / 8;
    float *sH = sm + Ly::oH, *sz = sm + Ly::oz, *sW = sm + Ly::oW, *sb = sm + Ly::ob;
    float *sphk = sm + Ly::ophk, *sv = sm + Ly::ov, *sq = sm + Ly::oq, *sphq = sm + Ly::ophq;
    float *sA = sm + Ly::oA, *sR = sm + Ly::oR, *sP = sm + Ly::oP;
    const int64_t kv = h / p.G;
    const int64_t unit = b * p.Hkv + kv;
    const int tid = threadIdx.x;
    const T* W = (const T*)a.Wf + kv * DH * (DF / 2);
    for (int e = tid; e < DH * (DF / 2); e += NT) sW[e] = ld(W + e);
    if (rec == nullptr) {
        for (int e = tid; e < DF * DH; e += NT) sH[e] = 0.0f;
        if (tid < DF) sz[tid] = 0.0f;
    } else {
        for (int e = tid; e < DF * DH; e += NT) sH[e] = rec[e];
        if (tid < DF) sz[tid] = rec[DF * DH + tid];
    }
    float tmax = kMinShift;
    for (int m = 0; m < p.M; ++m) tmax = fmaxf(tmax, a.sinks[h * p.M + m]);
    __syncthreads();

    const int r = tid >> 3, cs = tid & 7;
    const T* q = (const T*)a.q;
    const T* kk = (const T*)a.k;
    const T* vv = (const T*)a.v;
    for (int64_t i0 = s0; i0 < s1; i0 += TS) {
        const int n = (int)min64(TS, s1 - i0);
        gates_cumsum<T, DF, FAST>((const T*)a.g, b, p.L, p.Hkv, kv, i0, n, sb);
        // delayed stream: row t carries key/value i0 + t - w (absent before token w)
        const int rlo = (int)min64(n, max64(0, p.w - i0));
        load_rows<T, DH>(kk, b, p.L, p.Hkv, kv, i0 - p.w, rlo, n, sq, PH);
        load_rows<T, DH>(vv, b, p.L, p.Hkv, kv, i0 - p.w, rlo, n, sv, DH);
        __syncthreads();
        phi_rows<DH, DF, FAST>(sq, sW, sphk, rlo, n);
        __syncthreads();
        if (a.kdec != nullptr) {  // masked reading
            scale_entering_keys<DF, TS, NT, FAST>(sphk, a.kdec, b, p.L, p.Hkv, kv, i0 - p.w, rlo, n);
            __syncthreads();
        }
        load_rows<T, DH>(q, b, p.L, p.Hq, h, i0, 0, n, sq, PH);
        __syncthreads();
        phi_rows<DH, DF, FAST>(sq, sW, sphq, 0, n);
        __syncthreads();
        for (int e = tid; e < TS * DF; e += NT) {
            const int t = e / DF, f = e % DF;
            sR[t * PF + f] = sphq[t * PF + f] * ex<FAST>(sb[t * PF + f]);
        }
        __syncthreads();
        // state readout: phi(q_i) e^{b_i} . [H | z]
        float acc[NC], gden = 0.0f;
#pragma unroll
        for (int j = 0; j < NC; ++j) acc[j] = 0.0f;
        for (int f = 0; f < DF; ++f) {
            const float qt = sR[r * PF + f];
#pragma unroll
            for (int j = 0; j < NC; ++j) acc[j] = fmaf(qt, sH[f * DH + cs + 8 * j], acc[j]);
            gden = fmaf(qt, sz[f], gden);
        }
        // intra-sub-chunk state term: A_it = sum_f phq_if phk_tf e^{b_if - b_tf}, t <= i
        for (int e = tid; e < TS * TS; e += NT) {
            const int i = e / TS, t = e % TS;
            float val = 0.0f;
            if (t <= i && i < n && t >= rlo) {
                const float* qi = sphq + i * PF;
                const float* kt = sphk + t * PF;
                const float* bi = sb + i * PF;
                const float* bt = sb + t * PF;
                for (int f = 0; f < DF; ++f) val = fmaf(qi[f] * kt[f], ex<FAST>(bi[f] - bt[f]), val);
            }
            sA[i * (TS + 1) + t] = val;
        }
        __syncthreads();
        for (int t = 0; t < TS; ++t) {
            const float at = sA[r * (TS + 1) + t];
            gden += at;
#pragma unroll
            for (int j = 0; j < NC; ++j) acc[j] = fmaf(at, sv[t * DH + cs + 8 * j], acc[j]);
        }
        // window softmax over keys (i-w, i], online max, tiles of KT keys
        float mrun = tmax, l = 0.0f, wacc[NC];
#pragma unroll
        for (int j = 0; j < NC; ++j) wacc[j] = 0.0f;
        const int64_t i = i0 + r;
        const int64_t jlo = max64(0, i0 - p.w + 1), jhi = i0 + n - 1;
        float* sk = sR;
        float* sv2 = sR + KT * PH;
        for (int64_t j0 = jlo; j0 <= jhi; j0 += KT) {
            __syncthreads();
            for (int e = tid; e < KT * DH; e += NT) {
                const int t = e / DH, c = e % DH;
                const int64_t j = j0 + t;
                float kx = 0.0f, vx = 0.0f;
                if (j <= jhi) {
                    kx = ld(kk + ((b * p.L + j) * p.Hkv + kv) * DH + c);
                    vx = ld(vv + ((b * p.L + j) * p.Hkv + kv) * DH + c);
                }
                sk[t * PH + c] = kx;
                sv2[t * DH + c] = vx;
            }
            __syncthreads();
            float s[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int kx = cs + 8 * u;
                const int64_t j = j0 + kx;
                const bool valid = (r < n) && (j <= i) && (j > i - p.w) && (j <= jhi);
                float dot = 0.0f;
                const float* qr = sq + r * PH;
                const float* kr = sk + kx * PH;
                for (int c = 0; c < DH; ++c) dot = fmaf(qr[c], kr[c], dot);
                s[u] = valid ? dot * p.scale : -INFINITY;
            }
            float tm = fmaxf(s[0], s[1]);
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
            const float mnew = fmaxf(mrun, tm);
            const float corr = ex<FAST>(mrun - mnew);
            const float p0 = (s[0] == -INFINITY) ? 0.0f : ex<FAST>(s[0] - mnew);
            const float p1 = (s[1] == -INFINITY) ? 0.0f : ex<FAST>(s[1] - mnew);
            sP[r * KT + cs] = p0;
            sP[r * KT + cs + 8] = p1;
            float ps = p0 + p1;
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
            l = l * corr + ps;
#pragma unroll
            for (int j = 0; j < NC; ++j) wacc[j] *= corr;
            mrun = mnew;
            __syncwarp();
            for (int t = 0; t < KT; ++t) {
                const float pk = sP[r * KT + t];
#pragma unroll
                for (int j = 0; j < NC; ++j) wacc[j] = fmaf(pk, sv2[t * DH + cs + 8 * j], wacc[j]);
            }
        }
        // shared normaliser: y = (e^{-m} N_gla + N_win) / (e^{-m} D_gla + E_win + sum e^{t-m})
        if (r < n) {
            float ssum = 0.0f;
            for (int m = 0; m < p.M; ++m) ssum += ex<FAST>(a.sinks[h * p.M + m] - mrun);
            const float e = ex<FAST>(-mrun);
            const float den = e * gden + l + ssum;
            const float inv = 1.0f / den;
            T* yr = (T*)a.y + ((b * p.L + i) * p.Hq + h) * DH;
#pragma unroll
            for (int j = 0; j < NC; ++j) st(yr + cs + 8 * j, (e * acc[j] + wacc[j]) * inv);
            if (a.lse != nullptr && cs == 0) a.lse[(b * p.L + i) * p.Hq + h] = mrun + logf(den);
        }
        __syncthreads();
        state_update<DH, DF, FAST>(sH, sz, sphk, sv, sb);
    }
    if (a.S_out != nullptr && s1 == p.L && (h % p.G) == 0) {
        for (int e = tid; e < DF * DH; e += NT) a.S_out[unit * DF * DH + e] = sH[e];
        if (tid < DF && a.z_out != nullptr) a.z_out[unit * DF + tid] = sz[tid];
    }
}

template <typename T, int DH, int DF, bool FAST>
__global__ void __launch_bounds__(NT, 1) fwd_simt_main(Plan p, FwdArgs a) {
    extern __shared__ float sm[];
    const int64_t bh = blockIdx.x, seg = blockIdx.y;
    const int64_t b = bh / p.Hq, h = bh % p.Hq, kv = h / p.G;
    const int64_t s0 = seg * p.seg_len;
    if (s0 >= p.L) return;
    const int64_t s1 = min64(p.L, s0 + p.seg_len);
    const int64_t unit = b * p.Hkv + kv;
    const float* rec =
        seg == 0 ? nullptr
                 : a.seg + ((size_t)seg * (size_t)(p.B * p.Hkv) + (size_t)unit) * p.rec_floats;
    walk_head<T, DH, DF, FAST>(p, a, b, h, s0, s1, rec, sm);
}

// The rest of a segment that the tensor-core main walk handed over at a step whose gates close
// too hard for its factored decays (Lizard summary sec. 2-C: the cumulative gate product of
// such a stretch underflows).  One CTA per (batch x KV head, segment) of the tensor-core plan:
// the CTA's record slot (slot seg * rec_step) holds the state before that step and, in its
// first log-decay word, the step (-1: the segment is complete).  The group's query heads are
// walked one after another from that state, with exact per-pair decays.
template <typename T, int DH, int DF, bool FAST>
__global__ void __launch_bounds__(NT, 1) fwd_simt_tail(Plan p, FwdArgs a) {
    extern __shared__ float sm[];
    grid_dep_wait();  // the main walk's marks and hand-off states
    const int64_t unit = blockIdx.x, seg = blockIdx.y;
    const int64_t b = unit / p.Hkv, kv = unit % p.Hkv;
    const float* ho =
        a.seg + ((size_t)(seg * p.rec_step) * (size_t)(p.B * p.Hkv) + (size_t)unit) * p.rec_floats;
    const int stop = __float_as_int(ho[DF * DH + DF]);
    if (stop < 0) return;
    const int64_t len = seq_len(p, b);
    const int64_t s0 = (int64_t)stop * TS;
    const int64_t s1 = min64(len, seg * p.seg_len + p.seg_len);
    if (p.cu == nullptr) {
        for (int64_t hh = 0; hh < p.G; ++hh) {
            walk_head<T, DH, DF, FAST>(p, a, b, kv * p.G + hh, s0, s1, ho, sm);
            __syncthreads();
        }
        return;
    }
    // a packed sequence is walked as batch 0 of a plan of its own length, on arrays that start
    // at its first row (and at its state and z slots)
    Plan ps = p;
    ps.cu = nullptr;
    ps.B = 1;
    ps.L = len;
    const int64_t r0 = seq_row0(p, b);
    FwdArgs as = a;
    as.q = (const T*)a.q + r0 * p.Hq * DH;
    as.k = (const T*)a.k + r0 * p.Hkv * DH;
    as.v = (const T*)a.v + r0 * p.Hkv * DH;
    as.g = (const T*)a.g + r0 * p.Hkv * DF;
    as.kdec = a.kdec != nullptr ? a.kdec + r0 * p.Hkv * DF : nullptr;
    as.y = (T*)a.y + r0 * p.Hq * DH;
    as.lse = a.lse != nullptr ? a.lse + r0 * p.Hq : nullptr;
    as.S_out = a.S_out != nullptr ? a.S_out + b * p.Hkv * DF * DH : nullptr;
    as.z_out = a.z_out != nullptr ? a.z_out + b * p.Hkv * DF : nullptr;
    for (int64_t hh = 0; hh < p.G; ++hh) {
        walk_head<T, DH, DF, FAST>(ps, as, 0, kv * p.G + hh, s0, s1, ho, sm);
        __syncthreads();
    }
}

template <typename T>
__global__ void ring_fill_kernel(Plan p, const T* k, const T* v, T* kc, T* vc) {
    const int64_t unit = blockIdx.y, b = unit / p.Hkv, kv = unit % p.Hkv;
    const int64_t len = seq_len(p, b);
    const int64_t nt = min64(len, p.w);
    if ((int64_t)blockIdx.x >= nt) return;  // (a shorter packed sequence)
    const int64_t t = len - nt + blockIdx.x;
    const int64_t slot = t % (p.w + 1);
    const int64_t r0 = seq_row0(p, b);
    for (int64_t c = threadIdx.x; c < p.d; c += blockDim.x) {
        const int64_t src = ((r0 + t) * p.Hkv + kv) * p.d + c;
        const int64_t dst = (unit * (p.w + 1) + slot) * p.d + c;
        if (kc != nullptr) kc[dst] = k[src];
        if (vc != nullptr) vc[dst] = v[src];
    }
}

template <typename T, int DH, int DF, bool FAST>
cudaError_t launch_impl(const Plan& p, const FwdArgs& a, cudaStream_t s) {
    using Ly = Lay<DH, DF>;
    const size_t smem = Ly::bytes;
    cudaError_t err;
    err = cudaFuncSetAttribute(fwd_simt_main<T, DH, DF, FAST>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(fwd_simt_seglocal<T, DH, DF, FAST>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const unsigned U = (unsigned)(p.B * p.Hkv);
    if (p.P > 1) {
        fwd_simt_seglocal<T, DH, DF, FAST><<<dim3(U, (unsigned)(p.P - 1)), NT, smem, s>>>(p, a);
        cudaError_t es = launch_seg_scan(p, a.seg, s);
        if (es != cudaSuccess) return es;
    }
    if (a.ev_before) cudaEventRecord(a.ev_before, s);
    fwd_simt_main<T, DH, DF, FAST>
        <<<dim3((unsigned)(p.B * p.Hq), (unsigned)p.P), NT, smem, s>>>(p, a);
    if (a.ev_after) cudaEventRecord(a.ev_after, s);
    return cudaGetLastError();
}

template <typename T, int DH, int DF, bool FAST>
cudaError_t states_impl(const Plan& p, const FwdArgs& a, cudaStream_t s) {
    using Ly = Lay<DH, DF>;
    const size_t smem = Ly::bytes;
    cudaError_t err = cudaFuncSetAttribute(fwd_simt_seglocal<T, DH, DF, FAST>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    if (p.P > 1) {
        const unsigned U = (unsigned)(p.B * p.Hkv);
        fwd_simt_seglocal<T, DH, DF, FAST><<<dim3(U, (unsigned)(p.P - 1)), NT, smem, s>>>(p, a);
        return launch_seg_scan(p, a.seg, s);
    }
    return cudaGetLastError();
}

template <typename T, bool FAST>
cudaError_t states_dims(const Plan& p, const FwdArgs& a, cudaStream_t s) {
    if (p.d == 128 && p.D == 128) return states_impl<T, 128, 128, FAST>(p, a, s);
    if (p.d == 128 && p.D == 64) return states_impl<T, 128, 64, FAST>(p, a, s);
    if (p.d == 64 && p.D == 128) return states_impl<T, 64, 128, FAST>(p, a, s);
    if (p.d == 64 && p.D == 64) return states_impl<T, 64, 64, FAST>(p, a, s);
    return cudaErrorInvalidValue;
}

template <typename T, bool FAST>
cudaError_t dispatch_dims(const Plan& p, const FwdArgs& a, cudaStream_t s) {
    if (p.d == 128 && p.D == 128) return launch_impl<T, 128, 128, FAST>(p, a, s);
    if (p.d == 128 && p.D == 64) return launch_impl<T, 128, 64, FAST>(p, a, s);
    if (p.d == 64 && p.D == 128) return launch_impl<T, 64, 128, FAST>(p, a, s);
    if (p.d == 64 && p.D == 64) return launch_impl<T, 64, 64, FAST>(p, a, s);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_fwd_simt(const Plan& p, const FwdArgs& a, cudaStream_t s) {
    if (p.dtype == LIZARD_F32) return dispatch_dims<float, false>(p, a, s);
    return dispatch_dims<__nv_bfloat16, true>(p, a, s);
}

cudaError_t launch_fwd_states(const Plan& p, const FwdArgs& a, cudaStream_t s) {
    if (p.dtype == LIZARD_F32) return states_dims<float, false>(p, a, s);
    return states_dims<__nv_bfloat16, true>(p, a, s);
}

cudaError_t launch_fwd_tail(const Plan& p, const FwdArgs& a, cudaStream_t s) {
    if (p.dtype != LIZARD_BF16 || p.d != 128 || p.D != 128) return cudaErrorInvalidValue;
    using Ly = Lay<128, 128>;
    auto kern = fwd_simt_tail<__nv_bfloat16, 128, 128, true>;
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Ly::bytes);
    if (e != cudaSuccess) return e;
    return launch_dependent(kern, dim3((unsigned)(p.B * p.Hkv), (unsigned)p.P), dim3(NT),
                            Ly::bytes, s, p, a);
}

cudaError_t launch_seg_scan(const Plan& p, float* seg, cudaStream_t s, bool dependent) {
    const unsigned nE = (unsigned)(p.D * p.d + p.D);
    const dim3 grid((nE + 255) / 256, (unsigned)(p.B * p.Hkv));
    if (dependent) return launch_dependent(fwd_seg_scan, grid, dim3(256), 0, s, p, seg);
    fwd_seg_scan<<<grid, 256, 0, s>>>(p, seg);
    return cudaGetLastError();
}

cudaError_t launch_ring_fill(const Plan& p, const void* k, const void* v, void* kc, void* vc,
                             cudaStream_t s) {
    const int64_t nt = p.L < p.w ? p.L : p.w;
    if (nt <= 0) return cudaSuccess;
    dim3 grid((unsigned)nt, (unsigned)(p.B * p.Hkv));
    if (p.dtype == LIZARD_F32)
        ring_fill_kernel<float><<<grid, 128, 0, s>>>(p, (const float*)k, (const float*)v,
                                                     (float*)kc, (float*)vc);
    else
        ring_fill_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(
            p, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, (__nv_bfloat16*)kc,
            (__nv_bfloat16*)vc);
    return cudaGetLastError();
}

}  // namespace lz
