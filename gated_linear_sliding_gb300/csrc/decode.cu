// Single-token decode step of the Lizard token mixer (sm_103a).
//
// Lizard summary (gist.science/ko/paper/2507.09025), sec. 2-A-1: inference keeps a
// constant-size state updated token by token instead of a growing KV cache;
// sec. 4: generation at 32K keeps constant memory.  One step at position pos:
//   S <- Gamma_pos (.) S + phi(k_{pos-w}) v_{pos-w}^T,  z likewise (pos >= w),
//   y  = [phi(q) S + sum_{j in (pos-w, pos]} e^{s q.k_j} v_j]
//      / [phi(q).z + sum_j e^{s q.k_j} + sum_m e^{t_m}],
// with k_{pos-w}, v_{pos-w} and the window read from a (w+1)-slot ring cache.
//
// The step is bound by HBM traffic on the fp32 state (read and write of
// D x d x 4 bytes per (batch, KV head)).  Each (batch, KV head) unit is one
// cluster of NS CTAs; CTA r owns columns [r d/NS, (r+1) d/NS) of S and of the
// outputs.  Every CTA reads the old z, so the cluster barrier orders those reads
// before CTA 0 writes the new z.
#include <cooperative_groups.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace lz {
namespace {

constexpr int NT = 256;
constexpr int NS = 4;  // CTAs (column slices) per unit = cluster size

template <typename T, int DH, int DF>
struct DecLay {
    static constexpr int CW = DH / NS;       // columns per CTA
    static constexpr int NRG = NT / CW;      // row groups
    static constexpr int RPT = DF / NRG;     // state rows per thread
    static constexpr int GMAX = 8;
    static constexpr int WMAX = 256;         // window keys staged per step
};

// phi of one row x (smem, DH floats) with Wf [DH, DF/2] from global; one warp.
template <typename T, int DH, int DF>
__device__ __forceinline__ void phi_warp(const float* x, const T* Wk, float* out) {
    constexpr int H = DF / 2, NJ = H / 32;
    const int lane = threadIdx.x & 31;
    float u[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) u[j] = 0.0f;
    for (int c = 0; c < DH; ++c) {
        const float xc = x[c];
#pragma unroll
        for (int j = 0; j < NJ; ++j) u[j] = fmaf(xc, ld(Wk + c * H + lane + 32 * j), u[j]);
    }
    float mx = u[0], mn = u[0];
#pragma unroll
    for (int j = 1; j < NJ; ++j) {
        mx = fmaxf(mx, u[j]);
        mn = fminf(mn, u[j]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    }
    float ep[NJ], en[NJ], sp = 0.0f, sn = 0.0f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        ep[j] = expf(u[j] - mx);
        en[j] = expf(mn - u[j]);
        sp += ep[j];
        sn += en[j];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        sp += __shfl_xor_sync(0xffffffffu, sp, o);
        sn += __shfl_xor_sync(0xffffffffu, sn, o);
    }
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        out[lane + 32 * j] = ep[j] / sp;
        out[H + lane + 32 * j] = en[j] / sn;
    }
}

template <typename T, int DH, int DF>
__global__ void __cluster_dims__(NS, 1, 1) __launch_bounds__(NT)
    decode_kernel(Plan p, DecodeArgs a) {
    using Ly = DecLay<T, DH, DF>;
    constexpr int CW = Ly::CW, NRG = Ly::NRG, RPT = Ly::RPT;
    __shared__ float sx[(Ly::GMAX + 1) * DH];
    __shared__ float sphi[(Ly::GMAX + 1) * DF];
    __shared__ float sgam[DF];
    __shared__ float sz[DF];
    __shared__ float sred[NRG * Ly::GMAX * CW];
    __shared__ float ss[Ly::GMAX * Ly::WMAX];
    __shared__ float srow[Ly::GMAX * 4];

    cg::cluster_group cluster = cg::this_cluster();
    const int sl = (int)cluster.block_rank();
    const int64_t unit = blockIdx.x / NS;
    const int64_t b = unit / p.Hkv, kv = unit % p.Hkv;
    const int G = (int)p.G;
    const int64_t w = p.w, R = w + 1, pos = a.pos;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = tid % CW, rg = tid / CW, c0 = sl * CW;
    const bool admit = pos >= w;

    // 1. this CTA's state slice, into registers
    float* Sg = a.S + unit * DF * DH;
    float sreg[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) sreg[i] = Sg[(rg + NRG * i) * DH + c0 + c];

    // 2. the new token's q heads, the key leaving the window, gates, old z
    const T* kc = (const T*)a.kc;
    const T* vc = (const T*)a.vc;
    for (int e = tid; e < G * DH; e += NT) {
        const int hh = e / DH, cc = e % DH;
        sx[e] = ld((const T*)a.q + (b * p.Hq + kv * G + hh) * DH + cc);
    }
    for (int e = tid; e < DH; e += NT)
        sx[G * DH + e] = admit ? ld(kc + (unit * R + (pos - w) % R) * DH + e) : 0.0f;
    for (int f = tid; f < DF; f += NT) {
        sgam[f] = sigmoidf_(ld((const T*)a.g + unit * DF + f));
        sz[f] = a.z[unit * DF + f];
    }
    __syncthreads();
    // every CTA of the cluster has read the old z before CTA 0 may overwrite it
    cluster.sync();

    // 3. feature maps of the G query heads and of the admitted key (one warp per row)
    const T* Wk = (const T*)a.Wf + kv * DH * (DF / 2);
    for (int row = warp; row <= G; row += NT / 32) {
        if (row == G && !admit) {
            for (int f = lane; f < DF; f += 32) sphi[G * DF + f] = 0.0f;
        } else {
            phi_warp<T, DH, DF>(sx + row * DH, Wk, sphi + row * DF);
        }
    }
    __syncthreads();

    // 4. state update of this slice (in place) and partial readouts phi(q).S
    const float ve = admit ? ld(vc + (unit * R + (pos - w) % R) * DH + c0 + c) : 0.0f;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int f = rg + NRG * i;
        const float sv = fmaf(sgam[f], sreg[i], sphi[G * DF + f] * ve);
        sreg[i] = sv;
        Sg[f * DH + c0 + c] = sv;
    }
    for (int hh = 0; hh < G; ++hh) {
        float part = 0.0f;
#pragma unroll
        for (int i = 0; i < RPT; ++i) part = fmaf(sphi[hh * DF + rg + NRG * i], sreg[i], part);
        sred[(rg * G + hh) * CW + c] = part;
    }
    __syncthreads();
    for (int f = tid; f < DF; f += NT) {
        const float zn = fmaf(sgam[f], sz[f], sphi[G * DF + f]);
        sz[f] = zn;
        if (sl == 0) a.z[unit * DF + f] = zn;
    }

    // 5. window scores s_hj = scale q_h.k_j, j in (pos-w, pos]; the newest key is the input
    const int64_t nkeys = min64(w, pos + 1);
    const int64_t jstart = pos - nkeys + 1;
    for (int64_t jj = warp; jj < nkeys; jj += NT / 32) {
        const int64_t j = jstart + jj;
        const T* krow = (j == pos) ? (const T*)a.k + unit * DH : kc + (unit * R + j % R) * DH;
        float kr[DH / 32];
#pragma unroll
        for (int e = 0; e < DH / 32; ++e) kr[e] = ld(krow + lane + 32 * e);
        for (int hh = 0; hh < G; ++hh) {
            float part = 0.0f;
#pragma unroll
            for (int e = 0; e < DH / 32; ++e) part = fmaf(sx[hh * DH + lane + 32 * e], kr[e], part);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if (lane == 0) ss[hh * Ly::WMAX + jj] = part * p.scale;
        }
    }
    __syncthreads();

    // 6. per head: shift m, window weights, state denominator, sink sum
    for (int hh = warp; hh < G; hh += NT / 32) {
        const int64_t h = kv * G + hh;
        float m = kMinShift;
        for (int mm = 0; mm < p.M; ++mm) m = fmaxf(m, a.sinks[h * p.M + mm]);
        for (int64_t jj = lane; jj < nkeys; jj += 32) m = fmaxf(m, ss[hh * Ly::WMAX + jj]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.0f;
        for (int64_t jj = lane; jj < nkeys; jj += 32) {
            const float pw = expf(ss[hh * Ly::WMAX + jj] - m);
            ss[hh * Ly::WMAX + jj] = pw;
            l += pw;
        }
        float gd = 0.0f;
        for (int f = lane; f < DF; f += 32) gd = fmaf(sphi[hh * DF + f], sz[f], gd);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            l += __shfl_xor_sync(0xffffffffu, l, o);
            gd += __shfl_xor_sync(0xffffffffu, gd, o);
        }
        float ssum = 0.0f;
        for (int mm = 0; mm < p.M; ++mm) ssum += expf(a.sinks[h * p.M + mm] - m);
        if (lane == 0) {
            srow[hh * 4 + 0] = m;
            srow[hh * 4 + 1] = l;
            srow[hh * 4 + 2] = gd;
            srow[hh * 4 + 3] = ssum;
        }
    }
    __syncthreads();

    // 7. outputs of this slice's columns
    for (int e = tid; e < G * CW; e += NT) {
        const int hh = e / CW, cc = e % CW;
        float num = 0.0f;
        for (int r2 = 0; r2 < NRG; ++r2) num += sred[(r2 * G + hh) * CW + cc];
        float wv = 0.0f;
        for (int64_t jj = 0; jj < nkeys; ++jj) {
            const int64_t j = jstart + jj;
            const T* vrow = (j == pos) ? (const T*)a.v + unit * DH : vc + (unit * R + j % R) * DH;
            wv = fmaf(ss[hh * Ly::WMAX + jj], ld(vrow + c0 + cc), wv);
        }
        const float m = srow[hh * 4 + 0];
        const float E = expf(-m);
        const float den = E * srow[hh * 4 + 2] + srow[hh * 4 + 1] + srow[hh * 4 + 3];
        st((T*)a.y + (b * p.Hq + kv * G + hh) * DH + c0 + cc, (E * num + wv) / den);
    }

    // 8. the new token joins the ring (slot pos mod (w+1), never read in this step)
    T* kco = (T*)a.kc;
    T* vco = (T*)a.vc;
    for (int cc = tid; cc < CW; cc += NT) {
        const int64_t dst = (unit * R + pos % R) * DH + c0 + cc;
        kco[dst] = ((const T*)a.k)[unit * DH + c0 + cc];
        vco[dst] = ((const T*)a.v)[unit * DH + c0 + cc];
    }
}

template <typename T, int DH, int DF>
cudaError_t launch_t(const Plan& p, const DecodeArgs& a, cudaStream_t s) {
    const unsigned grid = (unsigned)(p.B * p.Hkv * NS);
    decode_kernel<T, DH, DF><<<grid, NT, 0, s>>>(p, a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch(const Plan& p, const DecodeArgs& a, cudaStream_t s) {
    if (p.d == 128 && p.D == 128) return launch_t<T, 128, 128>(p, a, s);
    if (p.d == 128 && p.D == 64) return launch_t<T, 128, 64>(p, a, s);
    if (p.d == 64 && p.D == 128) return launch_t<T, 64, 128>(p, a, s);
    if (p.d == 64 && p.D == 64) return launch_t<T, 64, 64>(p, a, s);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode(const Plan& p, const DecodeArgs& a, cudaStream_t s) {
    if (p.dtype == LIZARD_F32) return dispatch<float>(p, a, s);
    return dispatch<__nv_bfloat16>(p, a, s);
}

}  // namespace lz
