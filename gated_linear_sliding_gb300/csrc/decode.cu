// Single-token decode step of the Lizard token mixer (sm_103a).
//
// Lizard summary (gist.science/ko/paper/2507.09025), sec. 2-A-1: inference keeps a
// constant-size state updated token by token instead of a growing KV cache;
// sec. 4: generation at 32K keeps constant memory.  One step at position pos (one position
// for the batch, or one per sequence read from device memory):
//   S <- Gamma_pos (.) S + phi(k_{pos-w}) v_{pos-w}^T,  z likewise (pos >= w),
//   y  = [phi(q) S + sum_{j in (pos-w, pos]} e^{s q.k_j} v_j]
//      / [phi(q).z + sum_j e^{s q.k_j} + sum_m e^{t_m}],
// with k_{pos-w}, v_{pos-w} and the window read from a (w+1)-slot ring cache.
//
// The step is bound by HBM traffic on the fp32 state (read and write of D x d x 4 bytes
// per (batch, KV head)).  One CTA owns one (batch, KV head) unit: at entry every thread
// issues its share of all loads at once (its slice of the state into registers; Wf, the
// key and value windows, the token and z into shared memory with cp.async), so the CTA
// pays one memory latency, then computes the feature maps, the state update and readout,
// the window softmax and the outputs from on-chip data, and writes the state back.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace lz {
namespace {

constexpr int NT = 256;
constexpr int GMAX = 8;  // query heads per KV head

__device__ __forceinline__ void cp16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

template <typename T, int DH, int DF, int WMAX>
struct DecLay {
    static constexpr int NRG = NT / DH;       // row groups of the state
    static constexpr int RPT = DF / NRG;      // consecutive state rows per thread
    static_assert(RPT % 4 == 0, "rows are read four at a time");
    static constexpr int E = (int)sizeof(T);  // bytes per element
    static constexpr int KROW = DH * E + 16;  // padded key row (bytes)
    // byte offsets of the dynamic shared memory
    static constexpr int oW = 0;                                 // Wf [DH][DF/2]
    static constexpr int oK = oW + DH * (DF / 2) * E;            // key window [WMAX][KROW]
    static constexpr int oV = oK + WMAX * KROW;                  // value window [WMAX][DH]
    static constexpr int oQ = oV + WMAX * DH * E;                // q rows, k_{pos-w} [G+1][DH]
    static constexpr int oVE = oQ + (GMAX + 1) * DH * E;         // v_{pos-w} [DH]
    static constexpr int oG = oVE + ((DH * E + 15) / 16) * 16;   // gate logits [DF]
    static constexpr int oZ = oG + ((DF * E + 15) / 16) * 16;    // old z [DF] fp32
    static constexpr int oX = oZ + DF * 4;                       // fp32 rows [G+1][DH]
    static constexpr int oPhi = oX + (GMAX + 1) * DH * 4;        // phi rows [G+1][DF]
    static constexpr int oU = oPhi + (GMAX + 1) * DF * 4;        // u rows [G+1][DF/2]
    static constexpr int oGam = oU + (GMAX + 1) * (DF / 2) * 4;  // gates [DF]
    static constexpr int oS = oGam + DF * 4;                     // window scores [G][WMAX]
    static constexpr int oRed = oS + GMAX * WMAX * 4;            // partials [NRG][G][DH]
    static constexpr int oRow = oRed + NRG * GMAX * DH * 4;      // per head m, l, den_gla, sinks
    static constexpr int oSk = oRow + GMAX * 4 * 4;              // sink logits [G][M]
    static constexpr int bytes = oSk + GMAX * 64 * 4;
};

template <typename T, int DH, int DF, int WMAX>
__global__ void __launch_bounds__(NT) decode_kernel(Plan p, DecodeArgs a) {
    using Ly = DecLay<T, DH, DF, WMAX>;
    constexpr int NRG = Ly::NRG, RPT = Ly::RPT, E = Ly::E, H2 = DF / 2;
    extern __shared__ __align__(16) unsigned char sm[];
    T* sW = (T*)(sm + Ly::oW);
    T* sQ = (T*)(sm + Ly::oQ);
    T* sVE = (T*)(sm + Ly::oVE);
    T* sG = (T*)(sm + Ly::oG);
    float* sZ = (float*)(sm + Ly::oZ);
    float* sX = (float*)(sm + Ly::oX);
    float* sPhi = (float*)(sm + Ly::oPhi);
    float* sU = (float*)(sm + Ly::oU);
    float* sGam = (float*)(sm + Ly::oGam);
    float* sS = (float*)(sm + Ly::oS);
    float* sRed = (float*)(sm + Ly::oRed);
    float* sRow = (float*)(sm + Ly::oRow);
    float* sSk = (float*)(sm + Ly::oSk);

    const int64_t unit = blockIdx.x;
    const int64_t b = unit / p.Hkv, kv = unit % p.Hkv;
    const int G = (int)p.G;
    const int64_t w = p.w, R = w + 1, pos = a.pos_dev != nullptr ? a.pos_dev[b] : a.pos;
    if (pos < 0) {  // a negative per-sequence position: recorded, the sequence is left untouched
        if (threadIdx.x == 0) report((WsHeader*)a.header, LIZARD_ERR_INVALID_ARG, 40);
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = tid % DH, rg = tid / DH;
    const bool admit = pos >= w;
    const int64_t nkeys = min64(w, pos + 1);
    const int64_t jstart = pos - nkeys + 1;
    const T* kc = (const T*)a.kc;
    const T* vc = (const T*)a.vc;
    const T* knew = (const T*)a.k + unit * DH;
    const T* vnew = (const T*)a.v + unit * DH;

    // 1. issue every load: the state rows of this thread to registers, the rest to shared memory
    float* Sg = a.S + unit * DF * DH;
    float sreg[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) sreg[i] = Sg[(rg * RPT + i) * DH + c];
    {
        const T* Wk = (const T*)a.Wf + kv * DH * H2;
        constexpr int nW = DH * H2 * E / 16;
        for (int e = tid; e < nW; e += NT) cp16((char*)sW + 16 * e, (const char*)Wk + 16 * e);
        constexpr int cpr = DH * E / 16;  // 16-byte chunks per row
        for (int e = tid; e < nkeys * cpr; e += NT) {
            const int64_t jj = e / cpr, ch = e % cpr;
            const int64_t j = jstart + jj;
            const bool cur = j == pos;
            const T* ks = cur ? knew : kc + (unit * R + j % R) * DH;
            const T* vs = cur ? vnew : vc + (unit * R + j % R) * DH;
            cp16(sm + Ly::oK + jj * Ly::KROW + 16 * ch, (const char*)ks + 16 * ch);
            cp16(sm + Ly::oV + jj * DH * E + 16 * ch, (const char*)vs + 16 * ch);
        }
        const T* qrow = (const T*)a.q + (b * p.Hq + kv * G) * DH;
        for (int e = tid; e < G * cpr; e += NT) cp16((char*)sQ + 16 * e, (const char*)qrow + 16 * e);
        if (admit) {
            const T* ke = kc + (unit * R + (pos - w) % R) * DH;
            const T* ve = vc + (unit * R + (pos - w) % R) * DH;
            for (int e = tid; e < cpr; e += NT) {
                cp16((char*)(sQ + G * DH) + 16 * e, (const char*)ke + 16 * e);
                cp16((char*)sVE + 16 * e, (const char*)ve + 16 * e);
            }
        }
        const T* gr = (const T*)a.g + unit * DF;
        for (int e = tid; e < DF * E / 16; e += NT) cp16((char*)sG + 16 * e, (const char*)gr + 16 * e);
        const float* zr = a.z + unit * DF;
        for (int e = tid; e < DF * 4 / 16; e += NT) cp16((char*)sZ + 16 * e, (const char*)zr + 16 * e);
    }
    // the sink logits of the group's heads (read in step 6)
    for (int e = tid; e < G * (int)p.M; e += NT) cp4(sSk + e, a.sinks + kv * G * p.M + e);
    cp_wait_all();
    __syncthreads();

    // 2. token rows to fp32, gates
    for (int e = tid; e < (G + 1) * DH; e += NT) {
        const int r = e / DH;
        sX[e] = (r < G || admit) ? ld(sQ + e) : 0.0f;
    }
    for (int f = tid; f < DF; f += NT) sGam[f] = sigmoidf_(ld(sG + f));
    __syncthreads();

    // 3. u = x Wf for the G query rows and the admitted key.  Lanes run over features, so a
    //    warp reads one contiguous row of Wf per column cc; the NQ thread groups split cc and
    //    their partial sums are added in a fixed order.
    {
        constexpr int NQ = NT / H2, CQ = DH / NQ;
        const int f = tid % H2, qd = tid / H2;
        float acc[GMAX + 1];
#pragma unroll
        for (int r = 0; r <= GMAX; ++r) acc[r] = 0.0f;
        for (int cc = qd * CQ; cc < (qd + 1) * CQ; cc += 4) {
            const float w0 = ld(sW + cc * H2 + f), w1 = ld(sW + (cc + 1) * H2 + f),
                        w2 = ld(sW + (cc + 2) * H2 + f), w3 = ld(sW + (cc + 3) * H2 + f);
#pragma unroll
            for (int r = 0; r <= GMAX; ++r)
                if (r <= G) {
                    const float4 x = *reinterpret_cast<const float4*>(sX + r * DH + cc);
                    acc[r] = fmaf(x.x, w0, fmaf(x.y, w1, fmaf(x.z, w2, fmaf(x.w, w3, acc[r]))));
                }
        }
        // partials [NQ][G+1][H2] in the score and readout-partial buffers (contiguous, both
        // unused until step 4)
        static_assert(GMAX * WMAX + NRG * GMAX * DH >= (GMAX + 1) * NT, "partials fit");
        static_assert(Ly::oRed == Ly::oS + GMAX * WMAX * 4, "contiguous");
        float* sUp = sS;
#pragma unroll
        for (int r = 0; r <= GMAX; ++r)
            if (r <= G) sUp[(qd * (G + 1) + r) * H2 + f] = acc[r];
        __syncthreads();
        for (int e = tid; e < (G + 1) * H2; e += NT) {
            float u = 0.0f;
#pragma unroll
            for (int q2 = 0; q2 < NQ; ++q2) u += sUp[q2 * (G + 1) * H2 + e];
            sU[e] = u;
        }
    }
    __syncthreads();
    // phi rows: one warp per row, [softmax(u), softmax(-u)]
    for (int r = warp; r <= G; r += NT / 32) {
        constexpr int NJ = H2 / 32;
        float u[NJ];
#pragma unroll
        for (int j = 0; j < NJ; ++j) u[j] = sU[r * H2 + lane + 32 * j];
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
        const bool zero = (r == G) && !admit;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            sPhi[r * DF + lane + 32 * j] = zero ? 0.0f : ep[j] / sp;
            sPhi[r * DF + H2 + lane + 32 * j] = zero ? 0.0f : en[j] / sn;
        }
    }
    __syncthreads();

    // 4. state update (rows [rg RPT, rg RPT + RPT) of column c) and partial readouts phi(q).S
    const float ve = admit ? ld(sVE + c) : 0.0f;
    const int f0 = rg * RPT;
#pragma unroll
    for (int i = 0; i < RPT; i += 4) {
        const float4 gm = *reinterpret_cast<const float4*>(sGam + f0 + i);
        const float4 pk = *reinterpret_cast<const float4*>(sPhi + G * DF + f0 + i);
        sreg[i] = fmaf(gm.x, sreg[i], pk.x * ve);
        sreg[i + 1] = fmaf(gm.y, sreg[i + 1], pk.y * ve);
        sreg[i + 2] = fmaf(gm.z, sreg[i + 2], pk.z * ve);
        sreg[i + 3] = fmaf(gm.w, sreg[i + 3], pk.w * ve);
    }
#pragma unroll
    for (int i = 0; i < RPT; ++i) Sg[(f0 + i) * DH + c] = sreg[i];
    for (int hh = 0; hh < G; ++hh) {
        float part = 0.0f;
#pragma unroll
        for (int i = 0; i < RPT; i += 4) {
            const float4 ph = *reinterpret_cast<const float4*>(sPhi + hh * DF + f0 + i);
            part = fmaf(ph.x, sreg[i], part);
            part = fmaf(ph.y, sreg[i + 1], part);
            part = fmaf(ph.z, sreg[i + 2], part);
            part = fmaf(ph.w, sreg[i + 3], part);
        }
        sRed[(rg * G + hh) * DH + c] = part;
    }
    // new z (written back by the CTA, which owns the unit)
    for (int f = tid; f < DF; f += NT) {
        const float zn = fmaf(sGam[f], sZ[f], sPhi[G * DF + f]);
        sZ[f] = zn;
        a.z[unit * DF + f] = zn;
    }

    // 5. window scores s_hj = scale q_h.k_j: one key per lane, 16-byte reads of the padded
    //    key rows (consecutive lanes land in distinct bank groups), q broadcast
    for (int e = tid; e < G * nkeys; e += NT) {
        const int hh = e / (int)nkeys, jj = e % (int)nkeys;
        const unsigned char* kr = sm + Ly::oK + jj * Ly::KROW;
        const float* x = sX + hh * DH;
        float acc = 0.0f;
        constexpr int EPC = 16 / E;  // elements per 16-byte chunk
#pragma unroll 4
        for (int ch = 0; ch < DH / EPC; ++ch) {
            const uint4 wv = *reinterpret_cast<const uint4*>(kr + 16 * ch);
            const T* kv8 = reinterpret_cast<const T*>(&wv);
#pragma unroll
            for (int e2 = 0; e2 < EPC; e2 += 4) {
                const float4 x4 = *reinterpret_cast<const float4*>(x + ch * EPC + e2);
                acc = fmaf(x4.x, ld(kv8 + e2), acc);
                acc = fmaf(x4.y, ld(kv8 + e2 + 1), acc);
                acc = fmaf(x4.z, ld(kv8 + e2 + 2), acc);
                acc = fmaf(x4.w, ld(kv8 + e2 + 3), acc);
            }
        }
        sS[hh * WMAX + jj] = acc * p.scale;
    }
    __syncthreads();

    // 6. per head: shift m, window weights, state denominator, sink sum (one warp per head)
    for (int hh = warp; hh < G; hh += NT / 32) {
        float m = kMinShift;
        for (int mm = 0; mm < p.M; ++mm) m = fmaxf(m, sSk[hh * p.M + mm]);
        for (int jj = lane; jj < nkeys; jj += 32) m = fmaxf(m, sS[hh * WMAX + jj]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.0f;
        for (int jj = lane; jj < nkeys; jj += 32) {
            const float pw = expf(sS[hh * WMAX + jj] - m);
            sS[hh * WMAX + jj] = pw;
            l += pw;
        }
        float gd = 0.0f;
        for (int f = lane; f < DF; f += 32) gd = fmaf(sPhi[hh * DF + f], sZ[f], gd);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            l += __shfl_xor_sync(0xffffffffu, l, o);
            gd += __shfl_xor_sync(0xffffffffu, gd, o);
        }
        float ssum = 0.0f;
        for (int mm = 0; mm < p.M; ++mm) ssum += expf(sSk[hh * p.M + mm] - m);
        if (lane == 0) {
            sRow[hh * 4 + 0] = m;
            sRow[hh * 4 + 1] = l;
            sRow[hh * 4 + 2] = gd;
            sRow[hh * 4 + 3] = ssum;
        }
    }
    __syncthreads();

    // 7. outputs: two adjacent columns of one head per item
    const T* sV = (const T*)(sm + Ly::oV);
    for (int e = tid; e < G * (DH / 2); e += NT) {
        const int hh = e / (DH / 2), cc = 2 * (e % (DH / 2));
        float num0 = 0.0f, num1 = 0.0f;
#pragma unroll
        for (int r2 = 0; r2 < NRG; ++r2) {
            num0 += sRed[(r2 * G + hh) * DH + cc];
            num1 += sRed[(r2 * G + hh) * DH + cc + 1];
        }
        float wv0 = 0.0f, wv1 = 0.0f;
        const float* ps = sS + hh * WMAX;
        int jj = 0;
        for (; jj + 4 <= nkeys; jj += 4) {
            const float4 p4 = *reinterpret_cast<const float4*>(ps + jj);
            const float pj[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                wv0 = fmaf(pj[k], ld(sV + (jj + k) * DH + cc), wv0);
                wv1 = fmaf(pj[k], ld(sV + (jj + k) * DH + cc + 1), wv1);
            }
        }
        for (; jj < nkeys; ++jj) {
            wv0 = fmaf(ps[jj], ld(sV + jj * DH + cc), wv0);
            wv1 = fmaf(ps[jj], ld(sV + jj * DH + cc + 1), wv1);
        }
        const float m = sRow[hh * 4 + 0];
        const float Em = expf(-m);
        const float inv = 1.0f / (Em * sRow[hh * 4 + 2] + sRow[hh * 4 + 1] + sRow[hh * 4 + 3]);
        T* yo = (T*)a.y + (b * p.Hq + kv * G + hh) * DH + cc;
        st(yo, (Em * num0 + wv0) * inv);
        st(yo + 1, (Em * num1 + wv1) * inv);
    }

    // 8. the new token joins the ring (slot pos mod (w+1), never read in this step), from its
    //    staged copy (the last key and value of the window)
    {
        constexpr int cpr = DH * E / 16;
        const unsigned char* kn = sm + Ly::oK + (nkeys - 1) * Ly::KROW;
        const unsigned char* vn = sm + Ly::oV + (nkeys - 1) * DH * E;
        char* kd = (char*)((T*)a.kc + (unit * R + pos % R) * DH);
        char* vd = (char*)((T*)a.vc + (unit * R + pos % R) * DH);
        for (int ch = tid; ch < cpr; ch += NT) {
            *reinterpret_cast<uint4*>(kd + 16 * ch) = *reinterpret_cast<const uint4*>(kn + 16 * ch);
            *reinterpret_cast<uint4*>(vd + 16 * ch) = *reinterpret_cast<const uint4*>(vn + 16 * ch);
        }
    }
}

template <typename T, int DH, int DF, int WMAX>
cudaError_t launch_w(const Plan& p, const DecodeArgs& a, cudaStream_t s) {
    using Ly = DecLay<T, DH, DF, WMAX>;
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<T, DH, DF, WMAX>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::bytes);
    if (e != cudaSuccess) return e;
    decode_kernel<T, DH, DF, WMAX><<<(unsigned)(p.B * p.Hkv), NT, Ly::bytes, s>>>(p, a);
    return cudaGetLastError();
}

// window capacity 64 keys for the usual w <= 64 (smaller shared-memory footprint), 256 otherwise
template <typename T, int DH, int DF>
cudaError_t launch_t(const Plan& p, const DecodeArgs& a, cudaStream_t s) {
    return p.w <= 64 ? launch_w<T, DH, DF, 64>(p, a, s) : launch_w<T, DH, DF, 256>(p, a, s);
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
