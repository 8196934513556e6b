// Kernels of the two other decay readings of the Lizard token mixer.
//
// Lizard summary (gist.science/ko/paper/2507.09025), sec. 2-A-1: a data-dependent gate
// Gamma = sigmoid(g) decays a constant-size state of the tokens that have left the window.
// The pages do not say which gates such a key has seen.  The default (delayed-key) reading
// weighs key j <= i - w at query i with prod_{s=j+w+1..i} Gamma_s; the library also runs
//   LAGGED  prod_{s=j+1..i-w} Gamma_s  = the delayed reading on the gates moved w tokens
//           later (Gamma'_s = Gamma_{s-w}), so every delayed-reading kernel runs it on a
//           moved copy of g and the backward moves dg back;
//   MASKED  prod_{s=j+1..i} Gamma_s    = the delayed reading with each entering key's phi
//           scaled by c_j = prod_{s=j+1..j+w} Gamma_s, the gates it saw in the window; the
//           forward and backward walks (tensor-core and SIMT) apply e^{kd_j}, kd_j = log c_j
//           from key_decay_tiled (windows up to 64) or key_decay_kernel.
// Decode keeps the gate logits of the window in a ring like the keys and values: the
// lagged step decays by the gate of token pos - w, the masked step admits token pos - w
// scaled by the product of the gates of pos - w + 1 .. pos.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace lz {
namespace {

// An open gate (sigmoid(30) rounds to 1 in fp32): the rows before w of a moved gate
// sequence only decay the empty state.
constexpr float kOpenGate = 30.0f;

template <typename T>
__device__ __forceinline__ uint4 open_chunk() {
    if constexpr (sizeof(T) == 2) {
        const uint32_t h = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(kOpenGate));
        const uint32_t w = h | (h << 16);
        return make_uint4(w, w, w, w);
    } else {
        const uint32_t w = __float_as_uint(kOpenGate);
        return make_uint4(w, w, w, w);
    }
}

// g' row i = g row i - w of the same sequence (i >= w), else an open gate.  One thread per
// 16-byte chunk of a token row (Hkv D contiguous elements); grid.y = sequence.
template <typename T>
__global__ void gate_lag_kernel(Plan p, const T* __restrict__ g, T* __restrict__ out) {
    const int64_t b = blockIdx.y;
    const int64_t len = seq_len(p, b), r0 = seq_row0(p, b);
    const int64_t per_row = p.Hkv * p.D * (int64_t)sizeof(T) / 16;
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= len * per_row) return;
    const int64_t i = e / per_row, c = e % per_row;
    const uint4 val = i >= p.w
                          ? reinterpret_cast<const uint4*>(g + (r0 + i - p.w) * p.Hkv * p.D)[c]
                          : open_chunk<T>();
    reinterpret_cast<uint4*>(out + (r0 + i) * p.Hkv * p.D)[c] = val;
}

// log sigmoid(x) = min(x, 0) - log(1 + u), u = e^{-|x|} in (0, 1], for the window sums of
// the masked reading: log(1 + u) = 2 artanh(s) with s = u / (2 + u) <= 1/3, from the odd
// power series artanh(s) = s + s^3/3 + s^5/5 + ... taken through s^15 (the first term left
// out is below 2e-9 of the sum).  No branch, so the independent evaluations of one thread
// interleave; its error is a few fp32 ulp of log(1 + u) plus that of the hardware
// exponential and quotient.
__device__ __forceinline__ float log_sigmoid_series(float x) {
    const float u = __expf(-fabsf(x));
    const float s = __fdividef(u, 2.0f + u);
    const float z = s * s;
    float q = 1.0f / 15.0f;
    q = fmaf(q, z, 1.0f / 13.0f);
    q = fmaf(q, z, 1.0f / 11.0f);
    q = fmaf(q, z, 1.0f / 9.0f);
    q = fmaf(q, z, 1.0f / 7.0f);
    q = fmaf(q, z, 1.0f / 5.0f);
    q = fmaf(q, z, 1.0f / 3.0f);
    q = fmaf(q, z, 1.0f);
    return fminf(x, 0.0f) - 2.0f * s * q;
}

// kd[j] = sum_{s=j+1..min(j+w, len-1)} log sigmoid(g_s), one column (KV head x feature) per
// thread.  Every term is <= 0, so a sum that only adds never cancels.  A run of n <= w rows
// [a, a+n) has every window (j, j+w] straddle M = a + w: kd_j = (sum over (j, M]) + (sum over
// (M, j+w]), the first grown downward from the middle run (a+n, M], the second upward from
// M (kept per row in shared memory), both compensated fp32 sums; w + n - 1 logarithms per n
// rows.  Threads of a block take consecutive columns, so every load and store of a row is
// contiguous.  grid.x = column blocks x row blocks of KJ, grid.y = sequence.
constexpr int KJ = 64;

// s += x with the rounding error carried in c (Kahan).
__device__ __forceinline__ void comp_add(float& s, float& c, float x) {
    const float y = x - c;
    const float t = s + y;
    c = (t - s) - y;
    s = t;
}

template <typename T>
__global__ void __launch_bounds__(128) key_decay_kernel(Plan p, const T* __restrict__ g,
                                                        float* __restrict__ kd) {
    __shared__ float up[KJ][128];  // the upward sums, row t of the run x thread
    const int64_t b = blockIdx.y;
    const int64_t len = seq_len(p, b), r0 = seq_row0(p, b);
    const int64_t HD = p.Hkv * p.D, ncb = (HD + 127) / 128;
    const int64_t cb = blockIdx.x % ncb, jb = blockIdx.x / ncb;
    const int64_t col = cb * 128 + threadIdx.x;
    const int64_t j0 = jb * KJ;
    if (col >= HD || j0 >= len) return;  // no block barrier below
    const int64_t j1 = min64(len, j0 + KJ), last = len - 1, w = p.w;
    const T* gc = g + r0 * HD + col;
    float* upc = &up[0][threadIdx.x];
    // each pass takes its gates KB rows at a time, every load of a batch issued first
    constexpr int KB = 16;
    for (int64_t a = j0; a < j1; a += w) {
        const int n = (int)min64(w, j1 - a);
        const int64_t M = a + w, top = min64(M, last);
        float us = 0.0f, uc = 0.0f;
        upc[0] = 0.0f;
        for (int t0 = 1; t0 < n; t0 += KB) {  // upward: gates M+1 .. M+n-1
            float x[KB];
#pragma unroll
            for (int k = 0; k < KB; ++k)
                x[k] = t0 + k < n && M + t0 + k <= last ? ld(gc + (M + t0 + k) * HD) : 0.0f;
#pragma unroll
            for (int k = 0; k < KB; ++k) {
                if (t0 + k >= n) break;
                if (M + t0 + k <= last) comp_add(us, uc, log_sigmoid_series(x[k]));
                upc[(t0 + k) * 128] = us;
            }
        }
        float ds = 0.0f, dc = 0.0f;
        for (int64_t s0 = a + n + 1; s0 <= top; s0 += KB) {  // the middle run a+n+1 .. M
            float x[KB];
#pragma unroll
            for (int k = 0; k < KB; ++k) x[k] = s0 + k <= top ? ld(gc + (s0 + k) * HD) : 0.0f;
#pragma unroll
            for (int k = 0; k < KB; ++k)
                if (s0 + k <= top) comp_add(ds, dc, log_sigmoid_series(x[k]));
        }
        for (int t0 = n - 1; t0 >= 0; t0 -= KB) {  // downward: gate a+t+1 joins row a+t
            float x[KB];
#pragma unroll
            for (int k = 0; k < KB; ++k)
                x[k] = t0 - k >= 0 && a + t0 - k + 1 <= last ? ld(gc + (a + t0 - k + 1) * HD) : 0.0f;
#pragma unroll
            for (int k = 0; k < KB; ++k) {
                const int t = t0 - k;
                if (t < 0) break;
                if (a + t + 1 <= last) comp_add(ds, dc, log_sigmoid_series(x[k]));
                kd[(r0 + a + t) * HD + col] = ds + upc[t * 128];
            }
        }
    }
}

// The same sums for windows of at most TW rows, from shared memory: a CTA copies rows
// (j0, j0 + TR - 1 + w] of TC columns of g in with asynchronous 16-byte copies (all in
// flight at once), takes their logarithms once (1 + (w - 1)/TR per output instead of about
// 2), then each thread takes a (column, run of w rows) pair through the two passes above.
// Needs HD a multiple of 16 bytes of T and g 16-byte aligned.  grid.x = column blocks x row
// blocks of TR, grid.y = sequence; 128 threads.
constexpr int TR = 256, TC = 32, TW = 64;
constexpr size_t kKeyTileSmem = sizeof(float) * ((TR + TW) * TC + TW * 128);

// Four consecutive elements of shared memory (8- or 16-byte aligned) as floats.
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}

template <typename T>
__global__ void __launch_bounds__(128) key_decay_tiled(Plan p, const T* __restrict__ g,
                                                       float* __restrict__ kd) {
    extern __shared__ __align__(16) float ksm[];
    float* lam = ksm;                  // [TR + w - 1][TC]: log sigmoid of row j0 + 1 + r
    float* up = ksm + (TR + TW) * TC;  // [TW][128]: upward sums of the thread's run
    // the raw rows: in place of their logarithms (fp32) or in the upward sums' space (bf16)
    T* stage = sizeof(T) == 4 ? reinterpret_cast<T*>(lam) : reinterpret_cast<T*>(up);
    const int64_t b = blockIdx.y;
    const int64_t len = seq_len(p, b), r0 = seq_row0(p, b);
    const int64_t HD = p.Hkv * p.D, ncb = (HD + TC - 1) / TC;
    const int64_t cb = blockIdx.x % ncb, jb = blockIdx.x / ncb;
    const int64_t j0 = jb * TR, c0 = cb * TC;
    if (j0 >= len) return;  // the whole block leaves together
    const int64_t j1 = min64(len, j0 + TR), last = len - 1, w = p.w;
    const int tid = threadIdx.x, nrow = (int)(TR + w - 1);
    // (1) the tile of logarithms; rows past the sequence's end and columns past HD hold 0
    {
        constexpr int CH = 16 / (int)sizeof(T), NCH = TC / CH;  // elements, chunks per row
        const T* gt = g + (r0 + j0 + 1) * HD + c0;
        for (int e = tid; e < nrow * NCH; e += 128) {
            const int r = e / NCH, ch = e % NCH;
            if (j0 + 1 + r <= last && c0 + ch * CH < HD)
                cp_async16(stage + r * TC + ch * CH, gt + (int64_t)r * HD + ch * CH);
        }
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        // four columns per thread (HD is a multiple of 4, so a quad is wholly in or out)
        for (int e = tid; e < nrow * (TC / 4); e += 128) {
            const int r = e / (TC / 4), c = 4 * (e % (TC / 4));
            float4 l = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (j0 + 1 + r <= last && c0 + c < HD) {
                const float4 x = ld4(stage + r * TC + c);
                l = make_float4(log_sigmoid_series(x.x), log_sigmoid_series(x.y),
                                log_sigmoid_series(x.z), log_sigmoid_series(x.w));
            }
            *reinterpret_cast<float4*>(lam + r * TC + c) = l;  // (fp32: the same elements)
        }
    }
    __syncthreads();
    // (2) runs [a, a + n) of w rows, kd_j = (sum over (j, a + w]) + (sum over (a + w, j + w])
    const int64_t nrun = (j1 - j0 + w - 1) / w;
    float* upt = up + tid;
    for (int64_t pr = tid; pr < nrun * TC; pr += 128) {
        const int c = (int)(pr % TC);
        const int64_t a = j0 + (pr / TC) * w;
        if (c0 + c >= HD) continue;
        const int n = (int)min64(w, j1 - a);
        const float* lc = lam + c;
        const int mrow = (int)(a + w - j0 - 1);  // tile row of gate a + w (= M)
        float us = 0.0f, uc = 0.0f;
        upt[0] = 0.0f;
#pragma unroll 8
        for (int t = 1; t < n; ++t) {  // upward: gates M+1 .. M+n-1
            comp_add(us, uc, lc[(mrow + t) * TC]);
            upt[t * 128] = us;
        }
        float ds = 0.0f, dc = 0.0f;
#pragma unroll 8
        for (int r = (int)(a - j0) + n; r <= mrow; ++r) comp_add(ds, dc, lc[r * TC]);  // middle
        float* out = kd + (r0 + a) * HD + c0 + c;
#pragma unroll 8
        for (int t = n - 1; t >= 0; --t) {  // downward: gate a+t+1 joins row a+t
            comp_add(ds, dc, lc[((int)(a - j0) + t) * TC]);
            out[(int64_t)t * HD] = ds + upt[t * 128];
        }
    }
}

// The gate-ring step of a MASKED or LAGGED decode: one CTA per (sequence, KV head) unit, RP
// threads per feature (thread = part * D + f).  The ring is read before the new gate row goes
// to slot pos mod (w+1) (the slots read are other slots).  The masked reading's sum over the
// window splits into RP contiguous runs of slots, added in a fixed order.
constexpr int RP = 4;

template <typename T>
__global__ void __launch_bounds__(RP * 128, 3)
decode_ring_kernel(Plan p, int64_t pos_all, const int64_t* pos_dev,
                   const T* __restrict__ g, T* __restrict__ gc, void* out) {
    __shared__ float part_sum[RP][128];
    grid_dep_launch();  // the decode step may be launched now (it waits for this grid's end)
    const int64_t unit = blockIdx.x, b = unit / p.Hkv;
    const int f = (int)(threadIdx.x % p.D), part = (int)(threadIdx.x / p.D);
    const int64_t pos = pos_dev != nullptr ? pos_dev[b] : pos_all;
    if (pos < 0) return;  // the decode kernel reports it and leaves the sequence untouched
    const int64_t w = p.w, R = w + 1, e = unit * p.D + f;
    T* gu = gc + unit * R * p.D + f;
    const T gnew = g[e];
    if (p.decay == LIZARD_DECAY_LAGGED) {
        // the step decays by the gate of token pos - w; before that the state is empty
        if (part == 0) {
            if (pos >= w) ((T*)out)[e] = gu[((pos - w) % R) * p.D];
            else st((T*)out + e, kOpenGate);
        }
    } else {
        // token pos - w enters scaled by prod_{s=pos-w+1..pos} Gamma_s: this thread sums the
        // slots of its run of tokens pos-w+1 .. pos-1, RB slots at a time with every load of
        // a batch issued before the first logarithm, stepping the slot without a division
        constexpr int RB = 8;
        float acc = 0.0f;
        if (pos >= w) {
            const int64_t n = w - 1, per = (n + RP - 1) / RP;
            const int64_t s0 = pos - w + 1 + part * per, s1 = min64(pos, s0 + per);
            int slot = s0 < s1 ? (int)(s0 % R) : 0;
            for (int64_t c0 = s0; c0 < s1; c0 += RB) {
                float x[RB];
#pragma unroll
                for (int k = 0; k < RB; ++k) {
                    x[k] = c0 + k < s1 ? ld(gu + (int64_t)slot * p.D) : 0.0f;
                    slot = slot + 1 == (int)R ? 0 : slot + 1;
                }
#pragma unroll
                for (int k = 0; k < RB; ++k)
                    if (c0 + k < s1) acc += log_sigmoid_series(x[k]);
            }
        }
        part_sum[part][f] = acc;
        __syncthreads();
        if (part == 0) {
            float tot = 0.0f;
            if (pos >= w) {
#pragma unroll
                for (int k = 0; k < RP; ++k) tot += part_sum[k][f];
                tot += log_sigmoid_series(ld(&gnew));
            }
            ((float*)out)[e] = tot;
        }
    }
    if (part == 0) gu[(pos % R) * p.D] = gnew;
}

template <typename T>
__global__ void gate_ring_fill_kernel(Plan p, const T* __restrict__ g, T* __restrict__ gc) {
    const int64_t unit = blockIdx.y, b = unit / p.Hkv, kv = unit % p.Hkv;
    const int64_t nt = min64(p.L, p.w);
    if ((int64_t)blockIdx.x >= nt) return;
    const int64_t t = p.L - nt + blockIdx.x;
    const int64_t slot = t % (p.w + 1);
    for (int64_t c = threadIdx.x; c < p.D; c += blockDim.x)
        gc[(unit * (p.w + 1) + slot) * p.D + c] = g[((b * p.L + t) * p.Hkv + kv) * p.D + c];
}

// Reverse cumulative sum of each column of key-side gate terms (rows past L - 1 - w are zero),
// in chunks of KS rows: first every chunk's total, then each chunk adds the totals of the
// chunks after it (last first) and scans its own rows in reverse.  Fixed order throughout.
constexpr int KS = 64;

__global__ void key_chunk_total_kernel(Plan p, const float* __restrict__ kk, float* __restrict__ kt) {
    const int64_t HD = p.Hkv * p.D, nch = (p.L + KS - 1) / KS;
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= p.B * nch * HD) return;
    const int64_t col = e % HD, r = e / HD, chunk = r % nch, b = r / nch;
    const int64_t j0 = chunk * KS, j1 = min64(min64(p.L, j0 + KS), p.L - p.w);
    // rows taken KB at a time, every load of a batch issued before the first addition
    constexpr int KB = 16;
    const float* x = kk + b * p.L * HD + col;
    float s = 0.0f;
    for (int64_t jt = j0; jt < j1; jt += KB) {
        float v[KB];
#pragma unroll
        for (int k = 0; k < KB; ++k) v[k] = jt + k < j1 ? x[(jt + k) * HD] : 0.0f;
#pragma unroll
        for (int k = 0; k < KB; ++k)
            if (jt + k < j1) s += v[k];
    }
    kt[e] = s;
}

__global__ void key_suffix_kernel(Plan p, float* __restrict__ kk, const float* __restrict__ kt) {
    const int64_t HD = p.Hkv * p.D, nch = (p.L + KS - 1) / KS;
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= p.B * nch * HD) return;
    const int64_t col = e % HD, r = e / HD, chunk = r % nch, b = r / nch;
    float run = 0.0f;
    for (int64_t c = nch - 1; c > chunk; --c) run += kt[(b * nch + c) * HD + col];
    const int64_t j0 = chunk * KS, j1 = min64(p.L, j0 + KS);
    float* x = kk + b * p.L * HD + col;
    // rows read KB at a time before any of them is overwritten: the loads of a batch are in
    // flight together instead of each waiting behind the store before it
    constexpr int KB = 16;
    for (int64_t jt = j1 - 1; jt >= j0; jt -= KB) {
        float v[KB];
#pragma unroll
        for (int k = 0; k < KB; ++k) v[k] = jt - k >= j0 ? x[(jt - k) * HD] : 0.0f;
#pragma unroll
        for (int k = 0; k < KB; ++k) {
            const int64_t j = jt - k;
            if (j >= j0) {
                if (j <= p.L - 1 - p.w) run += v[k];
                x[j * HD] = run;
            }
        }
    }
}

size_t elem(const Plan& p) { return p.dtype == LIZARD_F32 ? 4 : 2; }

}  // namespace

size_t reading_scratch_bytes(const Plan& p) {
    const size_t n = (size_t)(p.T > 0 ? p.T : p.B * p.L) * (size_t)(p.Hkv * p.D);
    if (p.decay == LIZARD_DECAY_LAGGED) return (n * elem(p) + 255) & ~(size_t)255;
    if (p.decay == LIZARD_DECAY_MASKED) return (n * 4 + 255) & ~(size_t)255;
    return 0;
}

size_t decode_scratch_bytes(const Plan& p) {
    const size_t n = (size_t)(p.B * p.Hkv * p.D);
    if (p.decay == LIZARD_DECAY_LAGGED) return (n * elem(p) + 255) & ~(size_t)255;
    if (p.decay == LIZARD_DECAY_MASKED) return (n * 4 + 255) & ~(size_t)255;
    return 0;
}

cudaError_t launch_gate_lag(const Plan& p, const void* g, void* out, cudaStream_t s) {
    const int64_t per_row = p.Hkv * p.D * (int64_t)elem(p) / 16;
    const dim3 grid((unsigned)((p.L * per_row + 255) / 256), (unsigned)p.B);
    if (p.dtype == LIZARD_F32)
        gate_lag_kernel<float><<<grid, 256, 0, s>>>(p, (const float*)g, (float*)out);
    else
        gate_lag_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(p, (const __nv_bfloat16*)g,
                                                            (__nv_bfloat16*)out);
    return cudaGetLastError();
}

cudaError_t launch_key_decay(const Plan& p, const void* g, float* kd, cudaStream_t s) {
    if (p.w <= TW && (p.Hkv * p.D * (int64_t)elem(p)) % 16 == 0 && ((uintptr_t)g & 15u) == 0) {
        const int64_t ncb = (p.Hkv * p.D + TC - 1) / TC, njb = (p.L + TR - 1) / TR;
        const dim3 grid((unsigned)(ncb * njb), (unsigned)p.B);
        auto k = p.dtype == LIZARD_F32 ? (void*)key_decay_tiled<float>
                                       : (void*)key_decay_tiled<__nv_bfloat16>;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kKeyTileSmem);
        if (e != cudaSuccess) return e;
        if (p.dtype == LIZARD_F32)
            key_decay_tiled<float><<<grid, 128, kKeyTileSmem, s>>>(p, (const float*)g, kd);
        else
            key_decay_tiled<__nv_bfloat16><<<grid, 128, kKeyTileSmem, s>>>(
                p, (const __nv_bfloat16*)g, kd);
        return cudaGetLastError();
    }
    const int64_t ncb = (p.Hkv * p.D + 127) / 128;
    const int64_t njb = (p.L + KJ - 1) / KJ;
    const dim3 grid((unsigned)(ncb * njb), (unsigned)p.B);
    if (p.dtype == LIZARD_F32)
        key_decay_kernel<float><<<grid, 128, 0, s>>>(p, (const float*)g, kd);
    else
        key_decay_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(p, (const __nv_bfloat16*)g, kd);
    return cudaGetLastError();
}

cudaError_t launch_decode_ring(const Plan& p, const DecodeArgs& a, void* out, cudaStream_t s) {
    if (p.D > 128) return cudaErrorInvalidValue;  // the per-part sums hold 128 features
    // (the lagged step copies one gate row per unit: one thread per feature)
    const unsigned grid = (unsigned)(p.B * p.Hkv),
                   block = (unsigned)((p.decay == LIZARD_DECAY_LAGGED ? 1 : RP) * p.D);
    if (p.dtype == LIZARD_F32)
        decode_ring_kernel<float><<<grid, block, 0, s>>>(p, a.pos, a.pos_dev, (const float*)a.g,
                                                         (float*)a.gc, out);
    else
        decode_ring_kernel<__nv_bfloat16><<<grid, block, 0, s>>>(
            p, a.pos, a.pos_dev, (const __nv_bfloat16*)a.g, (__nv_bfloat16*)a.gc, out);
    return cudaGetLastError();
}

cudaError_t launch_gate_ring_fill(const Plan& p, const void* g, void* gc, cudaStream_t s) {
    const dim3 grid((unsigned)min64(p.L, p.w), (unsigned)(p.B * p.Hkv));
    if (p.dtype == LIZARD_F32)
        gate_ring_fill_kernel<float><<<grid, 128, 0, s>>>(p, (const float*)g, (float*)gc);
    else
        gate_ring_fill_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(p, (const __nv_bfloat16*)g,
                                                                  (__nv_bfloat16*)gc);
    return cudaGetLastError();
}

size_t key_suffix_scratch_floats(const Plan& p) {
    return (size_t)(p.B * ((p.L + KS - 1) / KS) * p.Hkv * p.D);
}

cudaError_t launch_key_suffix(const Plan& p, float* kk, float* kt, cudaStream_t s) {
    const int64_t n = (int64_t)key_suffix_scratch_floats(p);
    key_chunk_total_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(p, kk, kt);
    key_suffix_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(p, kk, kt);
    return cudaGetLastError();
}

}  // namespace lz
