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

#include <cstddef>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"
#include "tc_util.cuh"

namespace lz {
namespace {

using namespace sm100;
using tc::kTimeout;

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
    // masked decay reading: the admitted key enters scaled by the product of the gates of
    // tokens pos - w + 1 .. pos (its log, per feature, from the gate-ring step)
    if (a.kdec != nullptr && admit) {
        for (int f = tid; f < DF; f += NT) sPhi[G * DF + f] *= expf(a.kdec[unit * DF + f]);
        __syncthreads();
    }

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

// ---------------------------------------------------------------------------------------
// Streaming decode step for the LLaMA-3-8B-shaped heads (bf16, d = D = 128, at most four query
// heads per KV head, w <= 64).  The step reads and writes the fp32 state, 64 KB per (batch, KV
// head) unit, and around it does about 190 K multiply-adds of small products per unit (u = x Wf,
// window scores, window values, the readout phi(q).S).  One CTA per SM walks its units (unit =
// CTA + i x grid) as a two-stage pipeline of 8-warp groups: the front group computes u, the
// window scores, the feature maps, the softmax and P V of unit i+1 while the back group updates
// the state of unit i, writes it straight back to global memory from registers (each warp store
// covers four whole 128-byte rows) and forms y.  They hand over through a double-buffered slot
// of shared memory (feature maps, gates, v_{pos-w}, the window values, e^{-m} and the
// normaliser), with mbarriers for each direction.  The copy engine brings everything in: the key
// and value rings and the query rows by tensor-map loads in two 64-column halves with the
// 128-byte swizzle (a row's 16-byte chunk c sits at chunk c ^ (row mod 8), so the eight rows an
// ldmatrix reads fall in distinct bank groups), the new token's rows, gate logits and z by plain
// bulk copies, and the state by four 32-column fp32 boxes with the same swizzle, two units
// ahead.  The products run as warp-level tensor-core MMAs (mma.sync): bf16 operands for u and
// the scores; P V with the probabilities rounded to bf16 (and the normaliser summing the same
// rounded values); tf32 for the readout, whose B fragments are the very state elements the lane has just updated,
// passed as fp32 bit patterns (the MMA reads their upper 19 bits).  Rows of the 16-row A
// fragments beyond the query heads are zero.
constexpr int ST = 512;      // threads: 16 warps, two groups of 8
constexpr int SG = 4;        // query heads per KV head, at most
constexpr int SW = 64;       // window, at most
constexpr int RH = 9216;     // one 64-column half of a ring: (w+1) rows of 128 bytes, 1 KB-rounded
// A unit's rows: the copy engine writes them, the front group alone reads them.
struct alignas(1024) StreamRows {
    uint8_t kr[2][RH];                // key ring halves (swizzled)
    uint8_t vr[2][RH];                // value ring halves
    uint8_t q[2][1024];               // query rows of the group, halves
    __nv_bfloat16 kn[128], vn[128];   // the new token (plain layout)
    __nv_bfloat16 gl[128];            // its gate logits
    float z[128];
};
// What the front group hands the back group for one unit.
struct StreamHand {
    float phi[SG + 1][136];   // feature maps: query heads, then k_{pos-w} (rows padded by 8)
    float gam[128];           // gates
    float ve[128];            // v_{pos-w} (zero before token w)
    float pv[SG][128];        // window values sum_j e^{s_j - m} v_j
    float row[SG][2];         // e^{-m}, 1 / denominator
};
struct StreamSmem {
    float S[2][4][128 * 32];       // states: four 32-column boxes of 128 rows each (swizzled)
    StreamRows rows[2];
    StreamHand hand[2];
    float u[SG + 1][64];           // front: x Wf of the query rows and k_{pos-w}
    float ps[SG][SW];              // front: window scores
    __nv_bfloat16 ph[SG][72];      // front: window probabilities (bf16)
    float rowf[SG][2];             // front: m, E_win + sinks
    float xp[SG][128];             // back: readout partials of features 64 .. 127
    __nv_bfloat16 zrow[128];       // zeros: the rows of fragments past the heads or the window
    uint64_t full_in[2], full_s[2], front_done[2], back_done[2];
    int abort;                     // set by a group that gave up waiting
};
constexpr size_t kStreamSmem = sizeof(StreamSmem) + 1024;
static_assert(kStreamSmem <= 232448, "shared memory budget");
static_assert(sizeof(StreamRows) % 1024 == 0 && offsetof(StreamRows, kr) % 1024 == 0 &&
                  offsetof(StreamRows, vr) % 1024 == 0 && offsetof(StreamRows, q) % 1024 == 0 &&
                  offsetof(StreamRows, kn) % 16 == 0 && offsetof(StreamRows, vn) % 16 == 0 &&
                  offsetof(StreamRows, gl) % 16 == 0 && offsetof(StreamRows, z) % 16 == 0,
              "row regions");
static_assert(offsetof(StreamSmem, rows) % 1024 == 0 && offsetof(StreamSmem, hand) % 16 == 0 &&
                  sizeof(StreamHand) % 16 == 0 && offsetof(StreamSmem, ph) % 16 == 0 &&
                  offsetof(StreamSmem, xp) % 16 == 0 &&
                  offsetof(StreamSmem, zrow) % 16 == 0 && offsetof(StreamSmem, u) % 16 == 0 &&
                  offsetof(StreamSmem, ps) % 16 == 0 && offsetof(StreamHand, pv) % 16 == 0 &&
                  offsetof(StreamHand, ve) % 16 == 0 && offsetof(StreamHand, gam) % 16 == 0,
              "scratch rows");

// Kernel parameters of the streaming step: tensor maps of the rings ([B Hkv (w+1)] rows of
// 128 bf16, box 64 x (w+1)), of the query rows ([B Hq] rows, box 64 x G) and of the state
// ([B Hkv 128] rows of 128 fp32, box 32 x 128).
struct StreamMaps {
    CUtensorMap kc, vc, q, S;
};

// A row of 64-column halves at h0 / h1 whose 16-byte chunks are XORed with x (the swizzled
// rings and query rows: x = row mod 8; the plain token rows and the zero row: x = 0).
struct SRow {
    uint32_t h0, h1, x;
};
__device__ __forceinline__ SRow srow_swz(const uint8_t* half0, const uint8_t* half1, int r) {
    return SRow{smem_u32(half0) + 128u * r, smem_u32(half1) + 128u * r, (uint32_t)(r & 7)};
}
__device__ __forceinline__ SRow srow_plain(const void* p) {
    return SRow{smem_u32(p), smem_u32(p) + 128u, 0u};
}
// shared address of the 16-byte chunk c (0..15: columns 8c .. 8c+7) of a row
__device__ __forceinline__ uint32_t chunk_addr(const SRow& r, int c) {
    return (c < 8 ? r.h0 : r.h1) + ((((uint32_t)c & 7u) ^ r.x) << 4);
}

// The front leader issues a unit's rings, query rows, token rows and z ...
__device__ __forceinline__ void stream_issue_in(const StreamMaps& mp, const Plan& p,
                                                const DecodeArgs& a, StreamRows& B, uint64_t* bar,
                                                int un) {
    const int Hkv = (int)p.Hkv, G = (int)p.G, R = (int)p.w + 1;
    const int b = un / Hkv, kv = un - b * Hkv;
    mbar_arrive_expect_tx(bar, (uint32_t)(512 * R + 256 * G + 3 * 256 + 512));
    for (int h = 0; h < 2; ++h) {
        tma_load_2d(B.kr[h], &mp.kc, bar, 64 * h, un * R);
        tma_load_2d(B.vr[h], &mp.vc, bar, 64 * h, un * R);
        tma_load_2d(B.q[h], &mp.q, bar, 64 * h, b * (int)p.Hq + kv * G);
    }
    bulk_load(B.kn, (const __nv_bfloat16*)a.k + (int64_t)un * 128, 256u, bar);
    bulk_load(B.vn, (const __nv_bfloat16*)a.v + (int64_t)un * 128, 256u, bar);
    bulk_load(B.gl, (const __nv_bfloat16*)a.g + (int64_t)un * 128, 256u, bar);
    bulk_load(B.z, a.z + (int64_t)un * 128, 512u, bar);
}
// ... and the back leader its state, four 32-column boxes.
__device__ __forceinline__ void stream_issue_s(const StreamMaps& mp, float (*S)[128 * 32],
                                               uint64_t* bar, int un) {
    mbar_arrive_expect_tx(bar, 65536u);
    for (int cg = 0; cg < 4; ++cg) tma_load_2d(S[cg], &mp.S, bar, 32 * cg, 128 * un);
}

// D += A B on a 16 x 8 tile: bf16 operands (K = 16) or tf32 operands (K = 8), fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_tf32_1688(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack2(__nv_bfloat16 lo, __nv_bfloat16 hi) {
    return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}
// Four 8 x 8 bf16 matrices from shared memory; lane l gives the row address of row l % 8 of
// matrix l / 8 (plain: lane gets row l / 4, columns 2 (l % 4), +1 of each; .trans: the transpose).
__device__ __forceinline__ void ldsm_x4(uint32_t* r, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t* r, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// Barrier of one 8-warp group (named barrier 1: front, 2: back); the _and form returns whether
// every thread passed true.
__device__ __forceinline__ void group_bar(int id) {
    asm volatile("bar.sync %0, 256;" ::"r"(id) : "memory");
}
__device__ __forceinline__ bool group_bar_and(int id, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, 256, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id)
        : "memory");
    return r != 0;
}
// Bounded wait for a phase, also given up when the other group has aborted.
__device__ __forceinline__ bool stream_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort != 0 || clock64() - t0 > kTimeout) return false;
    }
    return true;
}

// KEYF: the masked decay reading (the admitted key's phi scaled by a.kdec's factor); a
// separate instantiation, so the other readings' code is not touched by it.
template <bool KEYF>
__global__ void __launch_bounds__(ST, 1)
    decode_stream_kernel(Plan p, DecodeArgs a, const __grid_constant__ StreamMaps mp) {
    extern __shared__ uint8_t smem_raw[];
    StreamSmem& sm = *reinterpret_cast<StreamSmem*>(
        (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, tq = lane & 3;  // fragment row group and thread in group
    const int lr = lane & 7, lm = lane >> 3;  // ldmatrix: row and matrix this lane addresses
    const int U = (int)(p.B * p.Hkv);         // below 2^31 (checked by the host)
    const int G = (int)p.G, Hkv = (int)p.Hkv, Hq = (int)p.Hq;
    const int w = (int)p.w, R = w + 1;
    WsHeader* hdr = (WsHeader*)a.header;
    const int u0 = blockIdx.x, ustep = gridDim.x;
    if (u0 >= U) return;
    const int64_t* const pos_dev = a.pos_dev;
    const int64_t pos_all = a.pos;
    volatile int* abort_flag = &sm.abort;
    if (tid == 0) {
        prefetch_tmap(&mp.kc);
        prefetch_tmap(&mp.vc);
        prefetch_tmap(&mp.q);
        prefetch_tmap(&mp.S);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.full_in[i], 1);
            mbar_init(&sm.full_s[i], 1);
            mbar_init(&sm.front_done[i], 1);
            mbar_init(&sm.back_done[i], 1);
        }
        sm.abort = 0;
        fence_mbar_init();
    }
    if (tid < 64) reinterpret_cast<uint32_t*>(sm.zrow)[tid] = 0u;
    __syncthreads();
    // after a gate-ring step this grid may start while that step still runs: nothing it
    // wrote (the step's gates or key factors) is read before here
    grid_dep_wait();

    if (warp < 8) {
        // ================= front: rows in; u, scores, feature maps, softmax, P V =================
        uint32_t out_in = 0u;  // leader's row copies in flight, one bit per buffer
        if (tid == 0) {
            stream_issue_in(mp, p, a, sm.rows[0], &sm.full_in[0], u0);
            out_in = 1u;
            if (u0 + ustep < U) {
                stream_issue_in(mp, p, a, sm.rows[1], &sm.full_in[1], u0 + ustep);
                out_in |= 2u;
            }
        }
        __nv_bfloat16* const kcw = (__nv_bfloat16*)a.kc;
        __nv_bfloat16* const vcw = (__nv_bfloat16*)a.vc;
        const __nv_bfloat16* const wfg = (const __nv_bfloat16*)a.Wf;
        const int M = (int)p.M;
        const float scale = p.scale;
        // B fragments of Wf (columns 8 warp .. + 7, all 128 inputs), kept in registers for the
        // CTA's KV head (the same for all its units whenever the grid is a multiple of Hkv;
        // reloaded when it changes); per head, max(t_m, kMinShift) and sum_m e^{t_m - that max}
        uint32_t wb[8][2];
        int kv_w = -1;
        // softmax rows: warps 5 and 6, one head per half-warp
        float tm = kMinShift, ts = 0.0f;  // of that head
        const int sh = warp == 5 || warp == 6 ? 2 * (warp - 5) + (lane >> 4) : -1;
        int it = 0;
        for (int un = u0; un < U; un += ustep, ++it) {
            const int sl = it & 1;
            const uint32_t par = (uint32_t)(it >> 1) & 1u;
            StreamRows& B = sm.rows[sl];
            StreamHand& H = sm.hand[sl];
            const int b = un / Hkv, kv = un - b * Hkv;
            if (kv != kv_w) {
                const __nv_bfloat16* W = wfg + (int64_t)kv * 128 * 64 + 8 * warp + gq;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const int k0 = 16 * ks + 2 * tq;
                    wb[ks][0] = pack2(W[k0 * 64], W[(k0 + 1) * 64]);
                    wb[ks][1] = pack2(W[(k0 + 8) * 64], W[(k0 + 9) * 64]);
                }
                if (sh >= 0) {
                    // the head's sinks spread over its half-warp: one load per lane, then
                    // max and sum across the 16 lanes
                    const float* t = a.sinks + (int64_t)(kv * G + sh) * M;
                    const int l = lane & 15;
                    float tv[4];
                    float mx = kMinShift;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {  // M <= 64 on this path
                        const int mm = l + 16 * k;
                        tv[k] = sh < G && mm < M ? t[mm] : -INFINITY;
                        mx = fmaxf(mx, tv[k]);
                    }
#pragma unroll
                    for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    float se = 0.0f;
#pragma unroll
                    for (int k = 0; k < 4; ++k) se += expf(tv[k] - mx);
#pragma unroll
                    for (int o = 8; o > 0; o >>= 1) se += __shfl_xor_sync(0xffffffffu, se, o);
                    tm = mx;
                    ts = sh < G ? se : 0.0f;
                }
                kv_w = kv;
            }
            const int64_t pos = pos_dev != nullptr ? pos_dev[b] : pos_all;
            bool okw = true;
            if (tid == 0) okw = stream_wait(&sm.full_in[sl], par, abort_flag);
            if (!group_bar_and(1, okw)) {
                if (tid == 0) {
                    report(hdr, LIZARD_ERR_TIMEOUT, 42);
                    sm.abort = 1;
                }
                break;
            }
            if (tid == 0) out_in &= ~(1u << sl);
            const bool run = pos >= 0;  // a negative per-sequence position: unit left untouched
            if (!run && tid == 0) report(hdr, LIZARD_ERR_INVALID_ARG, 43);
            const bool admit = pos >= w;
            const int nkeys = run ? (pos + 1 < w ? (int)pos + 1 : w) : 1;
            // masked decay reading: the log factors of the admitted key, loaded now for warp SG,
            // which forms that key's phi after the hand-off wait below
            float kl[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (KEYF && warp == SG && run && admit) {
                const float* kr2 = a.kdec + (int64_t)un * 128;
                kl[0] = kr2[lane];
                kl[1] = kr2[lane + 32];
                kl[2] = kr2[64 + lane];
                kl[3] = kr2[96 + lane];
            }
            // ring slots: the new token goes to slot_n = pos mod (w+1); the key that leaves the
            // window (token pos - w) sits in the slot after it; key jj of the window (token
            // pos - nkeys + 1 + jj) in slot (slot0 + jj) mod (w+1), the last being the new token
            const int slot_n = run ? (pos <= 0x7fffffff ? (int)pos % R : (int)(pos % R)) : 0;
            const int slot_e = slot_n + 1 == R ? 0 : slot_n + 1;
            const int slot0 =
                slot_n - (nkeys - 1) < 0 ? slot_n - (nkeys - 1) + R : slot_n - (nkeys - 1);
            const uint32_t zb = smem_u32(sm.zrow);
            // row of window key jj (the new token's own row for the last key; keys past the
            // window read the zero row, at chunks that keep the eight rows in distinct banks)
            auto key_row = [&](const uint8_t (*ring)[RH], const __nv_bfloat16* cur, int jj) {
                int sl2 = slot0 + jj;
                if (sl2 >= R) sl2 -= R;
                return jj < nkeys - 1 ? srow_swz(ring[0], ring[1], sl2)
                       : jj == nkeys - 1 ? srow_plain(cur)
                                         : SRow{zb, zb + 128u, (uint32_t)(jj & 7)};
            };
            if (run) {
                // u = x Wf (columns 8 warp .. + 7) and the window scores of keys 8 warp .. + 7,
                // both from the same A fragments: query rows 0..G-1, row SG the key that leaves
                // (zero before token w), zero rows elsewhere
                const SRow ar = lr < G ? srow_swz(B.q[0], B.q[1], lr)
                                : (lr == SG && admit) ? srow_swz(B.kr[0], B.kr[1], slot_e)
                                                      : SRow{zb, zb + 128u, (uint32_t)lr};
                const SRow kr = key_row(B.kr, B.kn, 8 * warp + lr);
                float du0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, du1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                float ds0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, ds1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int kp = 0; kp < 4; ++kp) {
                    uint32_t af[4], bf[4];
                    ldsm_x4(af, chunk_addr(ar, 4 * kp + lm));
                    ldsm_x4(bf, chunk_addr(kr, 4 * kp + lm));
                    mma_bf16_16816(du0, af[0], 0u, af[1], 0u, wb[2 * kp][0], wb[2 * kp][1]);
                    mma_bf16_16816(ds0, af[0], 0u, af[1], 0u, bf[0], bf[1]);
                    mma_bf16_16816(du1, af[2], 0u, af[3], 0u, wb[2 * kp + 1][0], wb[2 * kp + 1][1]);
                    mma_bf16_16816(ds1, af[2], 0u, af[3], 0u, bf[2], bf[3]);
                }
                if (gq <= SG)
                    *reinterpret_cast<float2*>(&sm.u[gq][8 * warp + 2 * tq]) =
                        make_float2(du0[0] + du1[0], du0[1] + du1[1]);
                if (gq < SG) {
                    const int j0 = 8 * warp + 2 * tq;
                    const bool hv = gq < G;
                    *reinterpret_cast<float2*>(&sm.ps[gq][j0]) =
                        make_float2(hv && j0 < nkeys ? (ds0[0] + ds1[0]) * scale : -INFINITY,
                                    hv && j0 + 1 < nkeys ? (ds0[1] + ds1[1]) * scale : -INFINITY);
                }
            }
            // the hand-off slot must be free (the back group done with unit it - 2)
            bool okh = true;
            if (tid == 0 && it >= 2) okh = stream_wait(&sm.back_done[sl], par ^ 1u, abort_flag);
            if (!group_bar_and(1, okh)) {
                if (tid == 0) {
                    report(hdr, LIZARD_ERR_TIMEOUT, 45);
                    sm.abort = 1;
                }
                break;
            }
            if (run) {
                if (warp <= SG) {
                    // feature maps: warps 0..3 the query heads, warp 4 the key that leaves
                    const int x = warp;
                    const float u0v = sm.u[x][lane], u1v = sm.u[x][lane + 32];
                    float mx = fmaxf(u0v, u1v), mn = fminf(u0v, u1v);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
                    }
                    const float p0 = __expf(u0v - mx), p1 = __expf(u1v - mx);
                    const float n0 = __expf(mn - u0v), n1 = __expf(mn - u1v);
                    float sp = p0 + p1, sn = n0 + n1;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        sp += __shfl_xor_sync(0xffffffffu, sp, o);
                        sn += __shfl_xor_sync(0xffffffffu, sn, o);
                    }
                    const bool zero = (x == SG && !admit) || (x < SG && x >= G);
                    const float ip = zero ? 0.0f : 1.0f / sp, in = zero ? 0.0f : 1.0f / sn;
                    if (KEYF && x == SG) {  // the admitted key's factor (masked reading)
                        H.phi[x][lane] = p0 * ip * __expf(kl[0]);
                        H.phi[x][lane + 32] = p1 * ip * __expf(kl[1]);
                        H.phi[x][64 + lane] = n0 * in * __expf(kl[2]);
                        H.phi[x][96 + lane] = n1 * in * __expf(kl[3]);
                    } else {
                        H.phi[x][lane] = p0 * ip;
                        H.phi[x][lane + 32] = p1 * ip;
                        H.phi[x][64 + lane] = n0 * in;
                        H.phi[x][96 + lane] = n1 * in;
                    }
                }
                if (sh >= 0) {
                    // softmax of head sh over a half-warp (keys l, l + 16, l + 32, l + 48):
                    // shift, probabilities rounded to bf16 (the P V operand; the normaliser sums
                    // the same rounded values, so y stays a weighted mean of the window's v),
                    // their sum with the sinks'; heads beyond G get zero rows
                    const int l = lane & 15;
                    float sv[4], m = tm;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        sv[k] = sm.ps[sh][l + 16 * k];
                        m = fmaxf(m, sv[k]);
                    }
#pragma unroll
                    for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                    float es = 0.0f;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const __nv_bfloat16 e = __float2bfloat16_rn(sh < G ? __expf(sv[k] - m) : 0.0f);
                        sm.ph[sh][l + 16 * k] = e;
                        es += __bfloat162float(e);
                    }
#pragma unroll
                    for (int o = 8; o > 0; o >>= 1) es += __shfl_xor_sync(0xffffffffu, es, o);
                    if (l == 0) {
                        sm.rowf[sh][0] = m;
                        sm.rowf[sh][1] = es + ts * __expf(tm - m);  // window + sum_m e^{t_m - m}
                    }
                } else if (warp == 7) {
                    // the new token joins the ring (slot pos mod (w+1), read by no one here)
                    __nv_bfloat16* dst = (lane < 16 ? kcw : vcw) + ((int64_t)un * R + slot_n) * 128;
                    const __nv_bfloat16* src = lane < 16 ? B.kn : B.vn;
                    *reinterpret_cast<uint4*>(dst + 8 * (lane & 15)) =
                        *reinterpret_cast<const uint4*>(src + 8 * (lane & 15));
                }
                group_bar(1);
                // window values N[h][c] = sum_j P[h][j] V[j][c], columns 16 warp .. + 15 (two
                // n-tiles): V's B fragments by transposing ldmatrix (keys 32 kp + lane), P's A
                // fragments (rows 0..SG-1 the heads, the others zero) by plain ldmatrix; the two
                // k-steps of each ldmatrix accumulate apart
                {
                    float n0[2][4] = {}, n1[2][4] = {};
                    const uint32_t prh = lr < SG ? smem_u32(sm.ph[lr]) : zb + 16u * lr;
#pragma unroll
                    for (int kp = 0; kp < 2; ++kp) {
                        uint32_t bv0[4], bv1[4], ah[4];
                        const SRow vrow = key_row(B.vr, B.vn, 32 * kp + lane);
                        ldsm_x4_t(bv0, chunk_addr(vrow, 2 * warp));
                        ldsm_x4_t(bv1, chunk_addr(vrow, 2 * warp + 1));
                        ldsm_x4(ah, prh + 64 * kp + 16 * lm);
                        mma_bf16_16816(n0[0], ah[0], 0u, ah[1], 0u, bv0[0], bv0[1]);
                        mma_bf16_16816(n0[1], ah[0], 0u, ah[1], 0u, bv1[0], bv1[1]);
                        mma_bf16_16816(n1[0], ah[2], 0u, ah[3], 0u, bv0[2], bv0[3]);
                        mma_bf16_16816(n1[1], ah[2], 0u, ah[3], 0u, bv1[2], bv1[3]);
                    }
                    if (gq < SG) {
#pragma unroll
                        for (int t = 0; t < 2; ++t)
                            *reinterpret_cast<float2*>(&H.pv[gq][16 * warp + 8 * t + 2 * tq]) =
                                make_float2(n0[t][0] + n1[t][0], n0[t][1] + n1[t][1]);
                    }
                }
                if (warp < G) {
                    // phi(q).z with the new z = Gamma z + phi(k_{pos-w}), then e^{-m} and the
                    // reciprocal of the denominator
                    float dz = 0.0f;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int f = lane + 32 * k;
                        const float gm = 1.0f / (1.0f + __expf(-__bfloat162float(B.gl[f])));
                        dz = fmaf(H.phi[warp][f], fmaf(gm, B.z[f], H.phi[SG][f]), dz);
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) dz += __shfl_xor_sync(0xffffffffu, dz, o);
                    if (lane == 0) {
                        const float em = __expf(-sm.rowf[warp][0]);
                        H.row[warp][0] = em;
                        H.row[warp][1] = 1.0f / (em * dz + sm.rowf[warp][1]);
                    }
                } else if (warp == 4 || warp == 5) {
                    // gates and the new z (features 64 (warp - 4) + lane, + 32)
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int f = 64 * (warp - 4) + lane + 32 * k;
                        const float gm = 1.0f / (1.0f + __expf(-__bfloat162float(B.gl[f])));
                        H.gam[f] = gm;
                        a.z[(int64_t)un * 128 + f] = fmaf(gm, B.z[f], H.phi[SG][f]);
                    }
                } else if (warp == 6) {
                    // v_{pos-w} for the state update (columns 4 lane .. + 3)
                    float4 vf = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    if (admit) {
                        const SRow vrow = srow_swz(B.vr[0], B.vr[1], slot_e);
                        const int c = 4 * lane;
                        uint2 vv;
                        asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];"
                                     : "=r"(vv.x), "=r"(vv.y)
                                     : "r"(chunk_addr(vrow, c >> 3) + 2 * (c & 7)));
                        const __nv_bfloat162 v01 = *reinterpret_cast<const __nv_bfloat162*>(&vv.x);
                        const __nv_bfloat162 v23 = *reinterpret_cast<const __nv_bfloat162*>(&vv.y);
                        vf = make_float4(__low2float(v01), __high2float(v01), __low2float(v23),
                                         __high2float(v23));
                    }
                    *reinterpret_cast<float4*>(&H.ve[4 * lane]) = vf;
                }
            }
            group_bar(1);  // the hand-off is written; this unit's rows are read
            if (tid == 0) {
                mbar_arrive(&sm.front_done[sl]);
                if (un + 2 * ustep < U) {
                    stream_issue_in(mp, p, a, B, &sm.full_in[sl], un + 2 * ustep);
                    out_in |= 1u << sl;
                }
            }
        }
        if (tid == 0 && *abort_flag != 0) {  // let row copies still in flight land
            for (int i = 0; i < 2; ++i)
                if (out_in & (1u << i)) {  // (one of the two parities is the copy in flight)
                    for (uint32_t ph = 0; ph < 2; ++ph) mbar_wait(&sm.full_in[i], ph, kTimeout / 8);
                }
        }
    } else {
        // ================= back: state in; update, readout, y; state out =================
        const int bt = tid - 256;  // thread within the group; 0 is the leader
        const int wq = warp - 8, cg = wq & 3, kh = wq >> 2;
        const int c0 = 32 * cg + 4 * gq;
        uint32_t out_s = 0u;  // leader's state copies in flight, one bit per buffer
        if (bt == 0) {
            stream_issue_s(mp, sm.S[0], &sm.full_s[0], u0);
            out_s = 1u;
            if (u0 + ustep < U) {
                stream_issue_s(mp, sm.S[1], &sm.full_s[1], u0 + ustep);
                out_s |= 2u;
            }
        }
        __nv_bfloat16* const yg = (__nv_bfloat16*)a.y;
        int it = 0;
        for (int un = u0; un < U; un += ustep, ++it) {
            const int sl = it & 1;
            const uint32_t par = (uint32_t)(it >> 1) & 1u;
            const StreamHand& H = sm.hand[sl];
            const int b = un / Hkv, kv = un - b * Hkv;
            const int64_t pos = pos_dev != nullptr ? pos_dev[b] : pos_all;
            const bool run = pos >= 0;
            bool okw = true;
            if (bt == 0)
                okw = stream_wait(&sm.front_done[sl], par, abort_flag) &&
                      stream_wait(&sm.full_s[sl], par, abort_flag);
            if (!group_bar_and(2, okw)) {
                if (bt == 0) {
                    report(hdr, LIZARD_ERR_TIMEOUT, 44);
                    sm.abort = 1;
                }
                break;
            }
            if (bt == 0) out_s &= ~(1u << sl);
            // S <- Gamma S + phi(k_{pos-w}) v_{pos-w}^T, written straight to global memory, and
            // the readout partials phi(q) S over features 64 kh .. + 63 for columns 32 cg .. + 31.
            // The lane holds columns 32 cg + 4 gq + j (the column gq of n-tile j) of feature rows
            // f = 64 kh + 8 ks + 2 tq and f + 1: one 16-byte chunk of each, at swizzled chunk
            // gq ^ (f mod 8), so each 8-lane phase of a 128-bit access reads 8 distinct chunks.
            // Those are exactly its B fragments (k = tq: feature f; k = tq + 4: f + 1) of the
            // tf32 products, passed as fp32 bit patterns.
            float acc[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
            if (run) {
                const float4 ve = *reinterpret_cast<const float4*>(&H.ve[c0]);
                const float* const Sq = sm.S[sl][cg];
                float* const Su = a.S + (int64_t)un * 128 * 128 + c0;
#pragma unroll 4
                for (int ks = 0; ks < 8; ++ks) {
                    const int f0 = 64 * kh + 8 * ks + 2 * tq, f1 = f0 + 1;
                    float4 s0 = *reinterpret_cast<const float4*>(Sq + f0 * 32 + ((gq ^ (2 * tq)) << 2));
                    float4 s1 =
                        *reinterpret_cast<const float4*>(Sq + f1 * 32 + ((gq ^ (2 * tq + 1)) << 2));
                    const float2 gg = *reinterpret_cast<const float2*>(&H.gam[f0]);
                    const float2 kk = *reinterpret_cast<const float2*>(&H.phi[SG][f0]);
                    s0.x = fmaf(gg.x, s0.x, kk.x * ve.x);
                    s0.y = fmaf(gg.x, s0.y, kk.x * ve.y);
                    s0.z = fmaf(gg.x, s0.z, kk.x * ve.z);
                    s0.w = fmaf(gg.x, s0.w, kk.x * ve.w);
                    s1.x = fmaf(gg.y, s1.x, kk.y * ve.x);
                    s1.y = fmaf(gg.y, s1.y, kk.y * ve.y);
                    s1.z = fmaf(gg.y, s1.z, kk.y * ve.z);
                    s1.w = fmaf(gg.y, s1.w, kk.y * ve.w);
                    *reinterpret_cast<float4*>(Su + f0 * 128) = s0;
                    *reinterpret_cast<float4*>(Su + f1 * 128) = s1;
                    const float2 qq = gq < SG ? *reinterpret_cast<const float2*>(&H.phi[gq][f0])
                                              : make_float2(0.0f, 0.0f);
                    const uint32_t a0 = __float_as_uint(qq.x), a2 = __float_as_uint(qq.y);
                    mma_tf32_1688(acc[0], a0, 0u, a2, 0u, __float_as_uint(s0.x), __float_as_uint(s1.x));
                    mma_tf32_1688(acc[1], a0, 0u, a2, 0u, __float_as_uint(s0.y), __float_as_uint(s1.y));
                    mma_tf32_1688(acc[2], a0, 0u, a2, 0u, __float_as_uint(s0.z), __float_as_uint(s1.z));
                    mma_tf32_1688(acc[3], a0, 0u, a2, 0u, __float_as_uint(s0.w), __float_as_uint(s1.w));
                }
                // C rows gq (heads): n = 2 tq of tile j is column 32 cg + 8 tq + j, n = 2 tq + 1
                // is column 32 cg + 8 tq + 4 + j; the upper feature half parks its partials
                if (kh == 1 && gq < SG) {
                    float* xo = &sm.xp[gq][32 * cg + 8 * tq];
                    *reinterpret_cast<float4*>(xo) =
                        make_float4(acc[0][0], acc[1][0], acc[2][0], acc[3][0]);
                    *reinterpret_cast<float4*>(xo + 4) =
                        make_float4(acc[0][1], acc[1][1], acc[2][1], acc[3][1]);
                }
            }
            group_bar(2);  // this state buffer is read; the partials are in
            if (bt == 0 && un + 2 * ustep < U) {
                stream_issue_s(mp, sm.S[sl], &sm.full_s[sl], un + 2 * ustep);
                out_s |= 1u << sl;
            }
            if (run && kh == 0 && gq < G) {
                // y = (e^{-m} phi(q) S + N) / denominator for head gq, columns 32 cg + 8 tq + j
                // and + 4 (j = 0..3), stored four bf16 at a time
                const float em = H.row[gq][0], inv = H.row[gq][1];
                const float* xo = &sm.xp[gq][32 * cg + 8 * tq];
                const float* nv = &H.pv[gq][32 * cg + 8 * tq];
                __nv_bfloat16* yo = yg + ((int64_t)b * Hq + kv * G + gq) * 128 + 32 * cg + 8 * tq;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const float4 xx = *reinterpret_cast<const float4*>(xo + 4 * hf);
                    const float4 nn = *reinterpret_cast<const float4*>(nv + 4 * hf);
                    const __nv_bfloat162 y01 =
                        __floats2bfloat162_rn(fmaf(em, acc[0][hf] + xx.x, nn.x) * inv,
                                              fmaf(em, acc[1][hf] + xx.y, nn.y) * inv);
                    const __nv_bfloat162 y23 =
                        __floats2bfloat162_rn(fmaf(em, acc[2][hf] + xx.z, nn.z) * inv,
                                              fmaf(em, acc[3][hf] + xx.w, nn.w) * inv);
                    uint2 pk;
                    pk.x = *reinterpret_cast<const uint32_t*>(&y01);
                    pk.y = *reinterpret_cast<const uint32_t*>(&y23);
                    *reinterpret_cast<uint2*>(yo + 4 * hf) = pk;
                }
            }
            group_bar(2);  // the hand-off slot and the partials are read
            if (bt == 0) mbar_arrive(&sm.back_done[sl]);
        }
        if (bt == 0 && *abort_flag != 0) {  // let state copies still in flight land
            for (int i = 0; i < 2; ++i)
                if (out_s & (1u << i)) {  // (one of the two parities is the copy in flight)
                    for (uint32_t ph = 0; ph < 2; ++ph) mbar_wait(&sm.full_s[i], ph, kTimeout / 8);
                }
        }
    }
}

bool aligned16(const void* ptr) { return ((uintptr_t)ptr & 15) == 0; }

// The streaming step takes the LLaMA-3-8B-shaped heads when every buffer it copies is 16-byte
// aligned and the tensor maps encode; otherwise the one-CTA-per-unit kernel runs.
bool decode_stream_plan(const Plan& p, const DecodeArgs& a, StreamMaps* mp) {
    if (!(p.dtype == LIZARD_BF16 && p.d == 128 && p.D == 128 && p.G >= 1 && p.G <= SG &&
          p.w >= 1 && p.w <= SW && p.M <= 64 && p.B * p.Hkv * (p.w + 1) < (int64_t)1 << 31 &&
          p.B * p.Hkv * 128 < (int64_t)1 << 31 && p.B * p.Hq < (int64_t)1 << 31))
        return false;
    if (!aligned16(a.kc) || !aligned16(a.vc) || !aligned16(a.q) || !aligned16(a.k) ||
        !aligned16(a.v) || !aligned16(a.g) || !aligned16(a.z) || !aligned16(a.S))
        return false;
    const cuuint64_t ring_dims[2] = {128, (cuuint64_t)(p.B * p.Hkv * (p.w + 1))};
    const cuuint64_t q_dims[2] = {128, (cuuint64_t)(p.B * p.Hq)};
    const cuuint64_t str[1] = {256};
    const cuuint32_t ring_box[2] = {64, (cuuint32_t)(p.w + 1)};
    const cuuint32_t q_box[2] = {64, (cuuint32_t)p.G};
    if (!(tc::make_map(&mp->kc, a.kc, 2, ring_dims, str, ring_box) &&
          tc::make_map(&mp->vc, a.vc, 2, ring_dims, str, ring_box) &&
          tc::make_map(&mp->q, a.q, 2, q_dims, str, q_box)))
        return false;
    auto fn = tc::encode_fn();
    const cuuint64_t s_dims[2] = {128, (cuuint64_t)(p.B * p.Hkv * 128)};
    const cuuint64_t s_str[1] = {512};
    const cuuint32_t s_box[2] = {32, 128};
    const cuuint32_t es[2] = {1, 1};
    return fn != nullptr &&
           fn(&mp->S, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.S, s_dims, s_str, s_box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_decode_stream(const Plan& p, const DecodeArgs& a, const StreamMaps& mp,
                                 cudaStream_t s) {
    int dev = 0, nsm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    auto kern = a.kdec != nullptr ? decode_stream_kernel<true> : decode_stream_kernel<false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kStreamSmem);
    if (e != cudaSuccess) return e;
    const int64_t U = p.B * p.Hkv;
    const unsigned grid = (unsigned)(U < nsm ? U : nsm);
    // after the other readings' gate-ring step: a dependent launch, overlapping its start
    if (p.decay != LIZARD_DECAY_DELAYED)
        return launch_dependent(kern, dim3(grid), dim3(ST), kStreamSmem, s, p, a, mp);
    kern<<<grid, ST, kStreamSmem, s>>>(p, a, mp);
    return cudaGetLastError();
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

cudaError_t launch_decode(const Plan& p, const DecodeArgs& a_in, cudaStream_t s) {
    DecodeArgs a = a_in;
    if (p.decay != LIZARD_DECAY_DELAYED) {
        // the gate-ring step: the lagged reading's decay gates (then the step runs as the
        // delayed one on them) or the masked reading's key factors, after the status word
        if (a.gc == nullptr) return cudaErrorInvalidValue;
        void* out = (char*)a.header + kHeaderBytes;
        const cudaError_t e = launch_decode_ring(p, a, out, s);
        if (e != cudaSuccess) return e;
        if (p.decay == LIZARD_DECAY_LAGGED) a.g = out;
        else a.kdec = (const float*)out;
    }
    StreamMaps mp;
    if (decode_stream_plan(p, a, &mp)) return launch_decode_stream(p, a, mp, s);
    if (p.dtype == LIZARD_F32) return dispatch<float>(p, a, s);
    return dispatch<__nv_bfloat16>(p, a, s);
}

}  // namespace lz
