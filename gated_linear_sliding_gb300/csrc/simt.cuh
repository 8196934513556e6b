// Block-wide building blocks of the SIMT kernels (forward, segment passes, backward):
// 256 threads walking a segment 32 tokens at a time with fp32 shared-memory tiles.
// Lizard summary (gist.science/ko/paper/2507.09025): sec. 2-C Hedgehog map, sec. 2-A-1
// log-space gates (decays as exp of differences of cumulative log-sigmoid gates).
#pragma once

#include "common.cuh"
#include "internal.h"

namespace lz {
namespace simt {

constexpr int NT = 256;  // threads per CTA
constexpr int TS = 32;   // tokens per sub-chunk
constexpr int KT = 16;   // window keys per smem tile

template <int DH, int DF>
struct Lay {
    static constexpr int PF = DF + 1;  // padded row strides (rows are read across lanes)
    static constexpr int PH = DH + 1;
    static constexpr int oH = 0;
    static constexpr int oz = oH + DF * DH;
    static constexpr int oW = oz + DF;
    static constexpr int ob = oW + DH * (DF / 2);
    static constexpr int ophk = ob + TS * PF;
    static constexpr int ov = ophk + TS * PF;
    static constexpr int oq = ov + TS * DH;
    static constexpr int ophq = oq + TS * PH;
    static constexpr int oA = ophq + TS * PF;
    static constexpr int oR = oA + TS * (TS + 1);
    static constexpr int RSZ = (TS * PF > KT * PH + KT * DH) ? TS * PF : KT * PH + KT * DH;
    static constexpr int oP = oR + RSZ;
    static constexpr int total = oP + TS * KT;
    static constexpr size_t bytes = sizeof(float) * (size_t)total;
};

// Rows t in [rlo, rhi) of x (token tok0 + t, head hx) into s[t][*] (stride sst); zeros elsewhere.
template <typename T, int DH>
__device__ __forceinline__ void load_rows(const T* x, int64_t b, int64_t L, int64_t Hx,
                                          int64_t hx, int64_t tok0, int rlo, int rhi, float* s,
                                          int sst) {
    for (int e = threadIdx.x; e < TS * DH; e += NT) {
        const int t = e / DH, c = e % DH;
        float val = 0.0f;
        if (t >= rlo && t < rhi) val = ld(x + ((b * L + tok0 + t) * Hx + hx) * DH + c);
        s[t * sst + c] = val;
    }
}

// Hedgehog map of TS rows: sout[t] = [softmax(x_t Wf), softmax(-x_t Wf)] for t in
// [rlo, rhi), zeros elsewhere.  Eight lanes per row.
template <int DH, int DF, bool FAST>
__device__ __forceinline__ void phi_rows(const float* sx, const float* sW, float* sout, int rlo,
                                         int rhi) {
    constexpr int H = DF / 2, PH = DH + 1, PF = DF + 1, NJ = H / 8;
    const int r = threadIdx.x >> 3, sub = threadIdx.x & 7;
    float u[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) u[j] = 0.0f;
    const float* x = sx + r * PH;
    for (int c = 0; c < DH; ++c) {
        const float xc = x[c];
        const float* wr = sW + c * H + sub;
#pragma unroll
        for (int j = 0; j < NJ; ++j) u[j] = fmaf(xc, wr[8 * j], u[j]);
    }
    float mx = u[0], mn = u[0];
#pragma unroll
    for (int j = 1; j < NJ; ++j) {
        mx = fmaxf(mx, u[j]);
        mn = fminf(mn, u[j]);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
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
    for (int o = 1; o < 8; o <<= 1) {
        sp += __shfl_xor_sync(0xffffffffu, sp, o);
        sn += __shfl_xor_sync(0xffffffffu, sn, o);
    }
    const bool valid = r >= rlo && r < rhi;
    const float ip = valid ? 1.0f / sp : 0.0f, in = valid ? 1.0f / sn : 0.0f;
    float* o = sout + r * PF;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        o[sub + 8 * j] = ep[j] * ip;
        o[H + sub + 8 * j] = en[j] * in;
    }
}

// sb[t][f] = sum_{s<=t} log sigmoid(g_{i0+s, f}) for the n valid rows; rows >= n add 0.
template <typename T, int DF, bool FAST>
__device__ __forceinline__ void gates_cumsum(const T* g, int64_t b, int64_t L, int64_t Hkv,
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

// Masked decay reading: the delayed keys of rows [rlo, n) (row t holds key tok0 + t of a
// sequence with L rows) enter the state with phi scaled by e^{kd}, kd = the log product of
// the w gates each key saw inside the window (rows of kd [B, L, Hkv, DF]).
template <int DF, int TSZ, int NTH, bool FAST>
__device__ __forceinline__ void scale_entering_keys(float* sphk, const float* kd, int64_t b,
                                                    int64_t L, int64_t Hkv, int64_t kv,
                                                    int64_t tok0, int rlo, int n) {
    constexpr int PF = DF + 1;
    for (int e = threadIdx.x; e < TSZ * DF; e += NTH) {
        const int t = e / DF, f = e % DF;
        if (t >= rlo && t < n) sphk[t * PF + f] *= ex<FAST>(kd[((b * L + tok0 + t) * Hkv + kv) * DF + f]);
    }
}

// H <- e^{b_last} (.) H + sum_t (phk_t e^{b_last - b_t}) v_t^T, z likewise.
// Overwrites sphk with the decayed keys.
template <int DH, int DF, bool FAST>
__device__ __forceinline__ void state_update(float* sH, float* sz, float* sphk, const float* sv,
                                             const float* sb) {
    constexpr int PF = DF + 1;
    for (int e = threadIdx.x; e < TS * DF; e += NT) {
        const int t = e / DF, f = e % DF;
        sphk[t * PF + f] *= ex<FAST>(sb[(TS - 1) * PF + f] - sb[t * PF + f]);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < DF * DH; e += NT) {
        const int f = e / DH, c = e % DH;
        float acc = ex<FAST>(sb[(TS - 1) * PF + f]) * sH[e];
#pragma unroll 8
        for (int t = 0; t < TS; ++t) acc = fmaf(sphk[t * PF + f], sv[t * DH + c], acc);
        sH[e] = acc;
    }
    if (threadIdx.x < DF) {
        const int f = threadIdx.x;
        float acc = ex<FAST>(sb[(TS - 1) * PF + f]) * sz[f];
        for (int t = 0; t < TS; ++t) acc += sphk[t * PF + f];
        sz[f] = acc;
    }
    __syncthreads();
}

}  // namespace simt
}  // namespace lz
