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
// CTA + i x grid) with two shared-memory buffers, so the copies of one unit overlap the compute
// of the one before.  Thread 0 moves all data with the copy engine: the key and value rings
// and the query rows by tensor-map loads in two 64-column halves with the 128-byte swizzle (a
// row's 16-byte chunk c sits at chunk c ^ (row mod 8), so the eight rows an ldmatrix reads fall
// in distinct bank groups), the new token's rows, gate logits and z by plain bulk copies, and
// the state by tensor-map copies of four 32-column fp32 boxes with the same swizzle, in and,
// once updated in place, out again (the stores drain while the next unit computes).  The copy
// engine takes requests in order, so a unit's loads are issued before the store ahead of them.  The products run as warp-level tensor-core MMAs (mma.sync):
// bf16 operands for u and the window scores; P V with the probabilities split into a bf16 head
// and tail (so they keep about 16 bits); tf32 for the readout, whose B fragments are the very
// state elements the lane has just updated, passed as fp32 bit patterns (the MMA reads their
// upper 19 bits).  Rows of the 16-row A fragments beyond the query heads are zero.
constexpr int ST = 512;      // threads: 16 warps
constexpr int SG = 4;        // query heads per KV head, at most
constexpr int SW = 64;       // window, at most
constexpr int RH = 9216;     // one 64-column half of a ring: (w+1) rows of 128 bytes, 1 KB-rounded
struct alignas(1024) StreamBuf {
    float S[4][128 * 32];             // state, columns 32 cg .. + 31 of all rows f (swizzled)
    uint8_t kr[2][RH];                // key ring halves (swizzled)
    uint8_t vr[2][RH];                // value ring halves
    uint8_t q[2][1024];               // query rows of the group, halves
    __nv_bfloat16 kn[128], vn[128];   // the new token (plain layout)
    __nv_bfloat16 gl[128];            // its gate logits
    float z[128];
};
struct StreamSmem {
    StreamBuf buf[2];
    float u[SG + 1][64];           // x Wf: query rows, then k_{pos-w}
    float phi[SG + 1][136];        // feature maps of the same rows (rows padded by 8 floats)
    float gam[128];
    float ps[SG][SW];              // window scores
    __nv_bfloat16 ph[SG][72];      // window probabilities, bf16 head ...
    __nv_bfloat16 pl[SG][72];      // ... and tail (p - head)
    float xp[4][SG][128];          // readout partials of the four feature quarters
    float pv[SG][128];             // window values
    float row[SG][4];              // m, E_win + sinks, e^{-m}, 1 / denominator
    __nv_bfloat16 zrow[128];       // zeros: the rows of fragments past the heads or the window
    uint64_t bar_in[2], bar_s[2];
};
constexpr size_t kStreamSmem = sizeof(StreamSmem) + 1024;
static_assert(kStreamSmem <= 232448, "shared memory budget");
static_assert(sizeof(StreamBuf) % 1024 == 0 && offsetof(StreamBuf, kr) % 1024 == 0 &&
                  offsetof(StreamBuf, vr) % 1024 == 0 && offsetof(StreamBuf, q) % 1024 == 0 &&
                  offsetof(StreamBuf, kn) % 16 == 0 && offsetof(StreamBuf, vn) % 16 == 0 &&
                  offsetof(StreamBuf, gl) % 16 == 0 && offsetof(StreamBuf, z) % 16 == 0,
              "buffer regions");
static_assert(offsetof(StreamSmem, ph) % 16 == 0 && offsetof(StreamSmem, pl) % 16 == 0 &&
                  offsetof(StreamSmem, xp) % 16 == 0 && offsetof(StreamSmem, pv) % 16 == 0 &&
                  offsetof(StreamSmem, zrow) % 16 == 0 && offsetof(StreamSmem, u) % 16 == 0 &&
                  offsetof(StreamSmem, ps) % 16 == 0 && (72 * 2) % 16 == 0,
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

// Thread 0 issues a unit's rings, query rows, token rows and z (no store reads them back, so
// the buffer is free once the unit's compute is done) ...
__device__ __forceinline__ void stream_issue_in(const StreamMaps& mp, const Plan& p,
                                                const DecodeArgs& a, StreamBuf& B, uint64_t* bar,
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
// ... and its state (once the store of the unit that used the buffer before has read it out).
__device__ __forceinline__ void stream_issue_s(const StreamMaps& mp, StreamBuf& B, uint64_t* bar,
                                               int un) {
    mbar_arrive_expect_tx(bar, 65536u);
    for (int cg = 0; cg < 4; ++cg) tma_load_2d(B.S[cg], &mp.S, bar, 32 * cg, 128 * un);
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
    float* const zg = a.z;
    __nv_bfloat16* const yg = (__nv_bfloat16*)a.y;
    __nv_bfloat16* const kcw = (__nv_bfloat16*)a.kc;
    __nv_bfloat16* const vcw = (__nv_bfloat16*)a.vc;
    const __nv_bfloat16* const wfg = (const __nv_bfloat16*)a.Wf;
    const float* const sinks = a.sinks;
    const int64_t* const pos_dev = a.pos_dev;
    const int64_t pos_all = a.pos;
    const int M = (int)p.M;
    const float scale = p.scale;
    if (tid == 0) {
        prefetch_tmap(&mp.kc);
        prefetch_tmap(&mp.vc);
        prefetch_tmap(&mp.q);
        prefetch_tmap(&mp.S);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.bar_in[i], 1);
            mbar_init(&sm.bar_s[i], 1);
        }
        fence_mbar_init();
        stream_issue_in(mp, p, a, sm.buf[0], &sm.bar_in[0], u0);
        stream_issue_s(mp, sm.buf[0], &sm.bar_s[0], u0);
        if (u0 + ustep < U) stream_issue_in(mp, p, a, sm.buf[1], &sm.bar_in[1], u0 + ustep);
    }
    if (tid < 64) reinterpret_cast<uint32_t*>(sm.zrow)[tid] = 0u;
    __syncthreads();
    uint32_t ph_in0 = 0u, ph_in1 = 0u, ph_s0 = 0u, ph_s1 = 0u;
    bool out_in0 = true, out_in1 = u0 + ustep < U, out_s0 = true, out_s1 = false;  // in flight
    bool ok = true, got = true, gs = true;
    int bi = 0;
    const SRow zr = srow_plain(sm.zrow);
    // warps 0..7: B fragments of Wf (columns 8 warp .. + 7, all 128 inputs), kept in registers
    // for the CTA's KV head (the same for all its units whenever the grid is a multiple of Hkv;
    // reloaded when it changes); per head, max(t_m, kMinShift) and sum_m e^{t_m - that max}
    uint32_t wb[8][2];
    int kv_w = -1;
    float tmx[SG], tse[SG];
    for (int un = u0; un < U; un += ustep, bi ^= 1) {
        StreamBuf& B = sm.buf[bi];
        StreamBuf& Bn = sm.buf[bi ^ 1];
        const int b = un / Hkv, kv = un - b * Hkv;
        if (kv != kv_w) {
            if (warp < 8) {
                const __nv_bfloat16* W = wfg + (int64_t)kv * 128 * 64 + 8 * warp + gq;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const int k0 = 16 * ks + 2 * tq;
                    wb[ks][0] = pack2(W[k0 * 64], W[(k0 + 1) * 64]);
                    wb[ks][1] = pack2(W[(k0 + 8) * 64], W[(k0 + 9) * 64]);
                }
            }
#pragma unroll
            for (int x = 0; x < SG; ++x) {
                float m = kMinShift, se = 0.0f;
                if (x < G) {
                    const float* t = sinks + (int64_t)(kv * G + x) * M;
                    for (int mm = 0; mm < M; ++mm) m = fmaxf(m, t[mm]);
                    for (int mm = 0; mm < M; ++mm) se += expf(t[mm] - m);
                }
                tmx[x] = m;
                tse[x] = se;
            }
            kv_w = kv;
        }
        const int64_t pos = pos_dev != nullptr ? pos_dev[b] : pos_all;
        // (1) everything but the state (one thread waits; the others wait at the barrier)
        if (tid == 0) got = mbar_wait(&sm.bar_in[bi], bi ? ph_in1 : ph_in0, kTimeout);
        if (!__syncthreads_and(got)) {
            if (tid == 0) report(hdr, LIZARD_ERR_TIMEOUT, 42);
            ok = false;
            break;
        }
        if (bi) ph_in1 ^= 1u;
        else ph_in0 ^= 1u;
        if (tid == 0) {
            if (bi) out_in1 = false;
            else out_in0 = false;
        }
        const bool run = pos >= 0;  // a negative per-sequence position leaves the unit untouched
        if (!run && tid == 0) report(hdr, LIZARD_ERR_INVALID_ARG, 43);
        const bool admit = pos >= w;
        const int nkeys = run ? (pos + 1 < w ? (int)pos + 1 : w) : 1;
        // ring slots: the new token goes to slot_n = pos mod (w+1); the key that leaves the
        // window (token pos - w) sits in the slot after it; key jj of the window (token
        // pos - nkeys + 1 + jj) in slot (slot0 + jj) mod (w+1), the last one being the new token
        const int slot_n = run ? (pos <= 0x7fffffff ? (int)pos % R : (int)(pos % R)) : 0;
        const int slot_e = slot_n + 1 == R ? 0 : slot_n + 1;
        const int slot0 = slot_n - (nkeys - 1) < 0 ? slot_n - (nkeys - 1) + R : slot_n - (nkeys - 1);
        // row of window key jj (the new token's own row for the last key; keys past the window
        // read the zero row)
        auto key_row = [&](const uint8_t (*ring)[RH], const __nv_bfloat16* cur, int jj) {
            int sl = slot0 + jj;
            if (sl >= R) sl -= R;
            return jj < nkeys - 1 ? srow_swz(ring[0], ring[1], sl)
                                  : jj == nkeys - 1 ? srow_plain(cur) : zr;
        };
        if (run) {
            // A fragments of the query rows (rows 0..G-1), row SG the key that leaves (zero
            // before token w), the others zero: two k-steps per ldmatrix
            const SRow ar = lr < G ? srow_swz(B.q[0], B.q[1], lr)
                          : (lr == SG && admit) ? srow_swz(B.kr[0], B.kr[1], slot_e) : zr;
            if (warp < 8) {
                // u = x Wf, columns 8 warp .. + 7
                float d0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, d1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int kp = 0; kp < 4; ++kp) {
                    uint32_t af[4];
                    ldsm_x4(af, chunk_addr(ar, 4 * kp + lm));
                    mma_bf16_16816(d0, af[0], 0u, af[1], 0u, wb[2 * kp][0], wb[2 * kp][1]);
                    mma_bf16_16816(d1, af[2], 0u, af[3], 0u, wb[2 * kp + 1][0], wb[2 * kp + 1][1]);
                }
                if (gq <= SG)
                    *reinterpret_cast<float2*>(&sm.u[gq][8 * warp + 2 * tq]) =
                        make_float2(d0[0] + d1[0], d0[1] + d1[1]);
                if (tid < 128) sm.gam[tid] = 1.0f / (1.0f + __expf(-__bfloat162float(B.gl[tid])));
            } else {
                // window scores of keys 8 (warp - 8) .. + 7 against the query rows
                const SRow kr = key_row(B.kr, B.kn, 8 * (warp - 8) + lr);
                float d0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, d1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int kp = 0; kp < 4; ++kp) {
                    uint32_t af[4], bf[4];
                    ldsm_x4(af, chunk_addr(ar, 4 * kp + lm));
                    ldsm_x4(bf, chunk_addr(kr, 4 * kp + lm));
                    mma_bf16_16816(d0, af[0], 0u, af[1], 0u, bf[0], bf[1]);
                    mma_bf16_16816(d1, af[2], 0u, af[3], 0u, bf[2], bf[3]);
                }
                if (gq < SG) {
                    const int j0 = 8 * (warp - 8) + 2 * tq;
                    const bool hv = gq < G;
                    *reinterpret_cast<float2*>(&sm.ps[gq][j0]) =
                        make_float2(hv && j0 < nkeys ? (d0[0] + d1[0]) * scale : -INFINITY,
                                    hv && j0 + 1 < nkeys ? (d0[1] + d1[1]) * scale : -INFINITY);
                }
            }
            __syncthreads();
            if (warp <= SG) {
                // feature maps: one warp per row (query heads, then the key that leaves)
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
                sm.phi[x][lane] = p0 * ip;
                sm.phi[x][lane + 32] = p1 * ip;
                sm.phi[x][64 + lane] = n0 * in;
                sm.phi[x][96 + lane] = n1 * in;
            } else if (warp >= 8 && warp < 8 + SG) {
                // per head: shift, probabilities (split into bf16 head and tail for P V), their
                // sum with the sinks'; heads beyond G get zero rows
                const int hh = warp - 8;
                const float tm = hh == 0 ? tmx[0] : hh == 1 ? tmx[1] : hh == 2 ? tmx[2] : tmx[3];
                const float ts = hh == 0 ? tse[0] : hh == 1 ? tse[1] : hh == 2 ? tse[2] : tse[3];
                const float s0 = sm.ps[hh][lane], s1 = sm.ps[hh][lane + 32];
                float m = fmaxf(tm, fmaxf(s0, s1));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                const float e0 = hh < G ? __expf(s0 - m) : 0.0f;
                const float e1 = hh < G ? __expf(s1 - m) : 0.0f;
                const __nv_bfloat16 h0 = __float2bfloat16_rn(e0), h1 = __float2bfloat16_rn(e1);
                sm.ph[hh][lane] = h0;
                sm.ph[hh][lane + 32] = h1;
                sm.pl[hh][lane] = __float2bfloat16_rn(e0 - __bfloat162float(h0));
                sm.pl[hh][lane + 32] = __float2bfloat16_rn(e1 - __bfloat162float(h1));
                float es = e0 + e1;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) es += __shfl_xor_sync(0xffffffffu, es, o);
                if (lane == 0) {
                    sm.row[hh][0] = m;
                    sm.row[hh][1] = es + ts * __expf(tm - m);  // window sum + sum_m e^{t_m - m}
                }
            }
            __syncthreads();
        }
        // the next unit's state goes to the other buffer once the store that buffer held (of
        // the unit before this one) has been read out
        if (tid == 0 && un + ustep < U) {
            bulk_wait_read();
            stream_issue_s(mp, Bn, &sm.bar_s[bi ^ 1], un + ustep);
            if (bi) out_s0 = true;
            else out_s1 = true;
        }
        if (run) {
            // (2) window values N[h][c] = sum_j P[h][j] V[j][c], columns 8 warp .. + 7: V's B
            //     fragments by transposing ldmatrix (keys 32 kp + lane), P's A fragments (rows
            //     0..SG-1 the heads, the others the zero row) by plain ldmatrix
            float nh[4] = {0.0f, 0.0f, 0.0f, 0.0f}, nl[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            const uint32_t prh = lr < SG ? smem_u32(sm.ph[lr]) : smem_u32(sm.zrow);
            const uint32_t prl = lr < SG ? smem_u32(sm.pl[lr]) : smem_u32(sm.zrow);
#pragma unroll
            for (int kp = 0; kp < 2; ++kp) {
                uint32_t bv[4], ah[4], al[4];
                ldsm_x4_t(bv, chunk_addr(key_row(B.vr, B.vn, 32 * kp + lane), warp));
                ldsm_x4(ah, prh + 64 * kp + 16 * lm);
                ldsm_x4(al, prl + 64 * kp + 16 * lm);
                mma_bf16_16816(nh, ah[0], 0u, ah[1], 0u, bv[0], bv[1]);
                mma_bf16_16816(nl, al[0], 0u, al[1], 0u, bv[0], bv[1]);
                mma_bf16_16816(nh, ah[2], 0u, ah[3], 0u, bv[2], bv[3]);
                mma_bf16_16816(nl, al[2], 0u, al[3], 0u, bv[2], bv[3]);
            }
            if (gq < SG)
                *reinterpret_cast<float2*>(&sm.pv[gq][8 * warp + 2 * tq]) =
                    make_float2(nh[0] + nl[0], nh[1] + nl[1]);
            // the new token joins the ring (slot pos mod (w+1), read by no one in this step)
            if (warp == 15) {
                __nv_bfloat16* dst = (lane < 16 ? kcw : vcw) + ((int64_t)un * R + slot_n) * 128;
                const __nv_bfloat16* src = lane < 16 ? B.kn : B.vn;
                *reinterpret_cast<uint4*>(dst + 8 * (lane & 15)) =
                    *reinterpret_cast<const uint4*>(src + 8 * (lane & 15));
            }
            // per head: phi(q).z with the new z = Gamma z + phi(k_{pos-w}), then e^{-m} and
            // the reciprocal of the denominator
            if (warp < G) {
                float dz = 0.0f;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int f = lane + 32 * k;
                    dz = fmaf(sm.phi[warp][f], fmaf(sm.gam[f], B.z[f], sm.phi[SG][f]), dz);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) dz += __shfl_xor_sync(0xffffffffu, dz, o);
                if (lane == 0) {
                    const float em = __expf(-sm.row[warp][0]);
                    sm.row[warp][2] = em;
                    sm.row[warp][3] = 1.0f / (em * dz + sm.row[warp][1]);
                }
            }
        }
        // (3) the state, S <- Gamma S + phi(k_{pos-w}) v_{pos-w}^T in place, and the readout
        //     partials phi(q) S over features 32 kg .. + 31 for columns 32 cg .. + 31.  The
        //     lane holds columns 32 cg + 4 gq + j (the column gq of n-tile j, j = 0..3) of
        //     feature rows f = 32 kg + 8 ks + 2 tq and f + 1: one 16-byte chunk of each, at
        //     swizzled chunk gq ^ (f mod 8), so each 8-lane phase of a 128-bit access reads 8
        //     distinct chunks.  Those are exactly its B fragments (k = tq, tq + 4; n = gq) of
        //     the tf32 products, with feature f for k = tq and f + 1 for k = tq + 4.
        if (tid == 0) gs = mbar_wait(&sm.bar_s[bi], bi ? ph_s1 : ph_s0, kTimeout);
        if (!__syncthreads_and(gs)) {
            if (tid == 0) report(hdr, LIZARD_ERR_TIMEOUT, 44);
            ok = false;
            break;
        }
        if (bi) ph_s1 ^= 1u;
        else ph_s0 ^= 1u;
        if (tid == 0) {
            if (bi) out_s1 = false;
            else out_s0 = false;
        }
        if (run) {
            const int cg = warp & 3, kg = warp >> 2;
            const int c0 = 32 * cg + 4 * gq;
            float ve[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (admit) {
                const SRow vrow = srow_swz(B.vr[0], B.vr[1], slot_e);
                uint2 vv;
                asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];"
                             : "=r"(vv.x), "=r"(vv.y)
                             : "r"(chunk_addr(vrow, c0 >> 3) + 2 * (c0 & 7)));
                const __nv_bfloat162 v01 = *reinterpret_cast<const __nv_bfloat162*>(&vv.x);
                const __nv_bfloat162 v23 = *reinterpret_cast<const __nv_bfloat162*>(&vv.y);
                ve[0] = __low2float(v01);
                ve[1] = __high2float(v01);
                ve[2] = __low2float(v23);
                ve[3] = __high2float(v23);
            }
            float acc[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
            float* const Sq = B.S[cg];
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const int f0 = 32 * kg + 8 * ks + 2 * tq, f1 = f0 + 1;
                float4* p0 = reinterpret_cast<float4*>(Sq + f0 * 32 + ((gq ^ (2 * tq)) << 2));
                float4* p1 = reinterpret_cast<float4*>(Sq + f1 * 32 + ((gq ^ (2 * tq + 1)) << 2));
                float4 s0 = *p0, s1 = *p1;
                const float2 gg = *reinterpret_cast<const float2*>(&sm.gam[f0]);
                const float2 kk = *reinterpret_cast<const float2*>(&sm.phi[SG][f0]);
                const float g0 = gg.x, g1 = gg.y, k0 = kk.x, k1 = kk.y;
                s0.x = fmaf(g0, s0.x, k0 * ve[0]);
                s0.y = fmaf(g0, s0.y, k0 * ve[1]);
                s0.z = fmaf(g0, s0.z, k0 * ve[2]);
                s0.w = fmaf(g0, s0.w, k0 * ve[3]);
                s1.x = fmaf(g1, s1.x, k1 * ve[0]);
                s1.y = fmaf(g1, s1.y, k1 * ve[1]);
                s1.z = fmaf(g1, s1.z, k1 * ve[2]);
                s1.w = fmaf(g1, s1.w, k1 * ve[3]);
                *p0 = s0;
                *p1 = s1;
                const float2 qq = gq < SG ? *reinterpret_cast<const float2*>(&sm.phi[gq][f0])
                                          : make_float2(0.0f, 0.0f);
                const uint32_t a0 = __float_as_uint(qq.x), a2 = __float_as_uint(qq.y);
                mma_tf32_1688(acc[0], a0, 0u, a2, 0u, __float_as_uint(s0.x), __float_as_uint(s1.x));
                mma_tf32_1688(acc[1], a0, 0u, a2, 0u, __float_as_uint(s0.y), __float_as_uint(s1.y));
                mma_tf32_1688(acc[2], a0, 0u, a2, 0u, __float_as_uint(s0.z), __float_as_uint(s1.z));
                mma_tf32_1688(acc[3], a0, 0u, a2, 0u, __float_as_uint(s0.w), __float_as_uint(s1.w));
            }
            // C rows gq (heads): n = 2 tq of tile j is column 32 cg + 8 tq + j, n = 2 tq + 1 is
            // column 32 cg + 8 tq + 4 + j
            if (gq < SG) {
                float* xo = &sm.xp[kg][gq][32 * cg + 8 * tq];
                *reinterpret_cast<float4*>(xo) = make_float4(acc[0][0], acc[1][0], acc[2][0], acc[3][0]);
                *reinterpret_cast<float4*>(xo + 4) = make_float4(acc[0][1], acc[1][1], acc[2][1], acc[3][1]);
            }
            if (tid < 128) zg[(int64_t)un * 128 + tid] = fmaf(sm.gam[tid], B.z[tid], sm.phi[SG][tid]);
        }
        fence_async_smem();  // the state's generic writes, before the copy engine reads them
        __syncthreads();
        if (tid == 0) {
            // this buffer's rows are free: the rows of the unit after next go in first, then
            // the state goes back (one thread, one bulk group)
            if (un + 2 * ustep < U) {
                stream_issue_in(mp, p, a, B, &sm.bar_in[bi], un + 2 * ustep);
                if (bi) out_in1 = true;
                else out_in0 = true;
            }
            if (run) {
                for (int cg = 0; cg < 4; ++cg) tma_store_2d(&mp.S, B.S[cg], 32 * cg, 128 * un);
                bulk_commit();
            }
        }
        if (!run) continue;  // the same for every thread; nothing else is written
        {  // y: one (head, column) per thread
            const int h = tid >> 7, c = tid & 127;
            if (h < G) {
                const float X = (sm.xp[0][h][c] + sm.xp[1][h][c]) + (sm.xp[2][h][c] + sm.xp[3][h][c]);
                yg[((int64_t)b * Hq + kv * G + h) * 128 + c] =
                    __float2bfloat16_rn(fmaf(sm.row[h][2], X, sm.pv[h][c]) * sm.row[h][3]);
            }
        }
        __syncthreads();  // the scratch rows are reused by the next unit
    }
    if (tid == 0) {
        bulk_wait_all();  // the last stores have completed
        if (!ok) {        // let copies still in flight land before the CTA exits
            if (out_in0) mbar_wait(&sm.bar_in[0], ph_in0, kTimeout);
            if (out_in1) mbar_wait(&sm.bar_in[1], ph_in1, kTimeout);
            if (out_s0) mbar_wait(&sm.bar_s[0], ph_s0, kTimeout);
            if (out_s1) mbar_wait(&sm.bar_s[1], ph_s1, kTimeout);
        }
    }
}

bool aligned16(const void* ptr) { return ((uintptr_t)ptr & 15) == 0; }

// The streaming step takes the LLaMA-3-8B-shaped heads when every buffer it copies is 16-byte
// aligned and the tensor maps encode; otherwise the one-CTA-per-unit kernel runs.
bool decode_stream_plan(const Plan& p, const DecodeArgs& a, StreamMaps* mp) {
    if (!(p.dtype == LIZARD_BF16 && p.d == 128 && p.D == 128 && p.G >= 1 && p.G <= SG &&
          p.w >= 1 && p.w <= SW && p.B * p.Hkv * (p.w + 1) < (int64_t)1 << 31 &&
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
    e = cudaFuncSetAttribute(decode_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kStreamSmem);
    if (e != cudaSuccess) return e;
    const int64_t U = p.B * p.Hkv;
    const unsigned grid = (unsigned)(U < nsm ? U : nsm);
    decode_stream_kernel<<<grid, ST, kStreamSmem, s>>>(p, a, mp);
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

cudaError_t launch_decode(const Plan& p, const DecodeArgs& a, cudaStream_t s) {
    StreamMaps mp;
    if (decode_stream_plan(p, a, &mp)) return launch_decode_stream(p, a, mp, s);
    if (p.dtype == LIZARD_F32) return dispatch<float>(p, a, s);
    return dispatch<__nv_bfloat16>(p, a, s);
}

}  // namespace lz
