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
//           from key_decay_kernel.
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

// kd[j] = sum_{s=j+1..min(j+w, len-1)} log sigmoid(g_s) for KJ consecutive rows j of one
// column (KV head x feature) per thread, a window sum slid one row at a time in fp64 (the
// per-gate logarithms in fp32).  Threads of a block take consecutive columns, so every load
// and store of a row is contiguous.  grid.x = column blocks x row blocks, grid.y = sequence.
constexpr int KJ = 64;

template <typename T>
__global__ void __launch_bounds__(128) key_decay_kernel(Plan p, const T* __restrict__ g,
                                                        float* __restrict__ kd) {
    const int64_t b = blockIdx.y;
    const int64_t len = seq_len(p, b), r0 = seq_row0(p, b);
    const int64_t HD = p.Hkv * p.D, ncb = (HD + 127) / 128;
    const int64_t cb = blockIdx.x % ncb, jb = blockIdx.x / ncb;
    const int64_t col = cb * 128 + threadIdx.x;
    const int64_t j0 = jb * KJ;
    if (col >= HD || j0 >= len) return;
    const int64_t j1 = min64(len, j0 + KJ), last = len - 1;
    const T* gc = g + r0 * HD + col;
    double acc = 0.0;
    for (int64_t s = j0 + 1; s <= min64(j0 + p.w, last); ++s)
        acc += (double)log_sigmoid<false>(ld(gc + s * HD));
#pragma unroll 4
    for (int64_t j = j0; j < j1; ++j) {
        kd[(r0 + j) * HD + col] = (float)acc;
        // the window of row j + 1 is s = j+2 .. j+1+w: gate j+1+w joins, gate j+1 leaves
        const float in = j + 1 + p.w <= last ? log_sigmoid<false>(ld(gc + (j + 1 + p.w) * HD)) : 0.0f;
        const float out = j + 1 <= last ? log_sigmoid<false>(ld(gc + (j + 1) * HD)) : 0.0f;
        acc += (double)in - (double)out;
    }
}

// The gate-ring step of a MASKED or LAGGED decode: one CTA per (sequence, KV head) unit, RP
// threads per feature (thread = part * D + f).  The ring is read before the new gate row goes
// to slot pos mod (w+1) (the slots read are other slots).  The masked reading's sum over the
// window splits into RP contiguous runs of slots, added in a fixed order.
constexpr int RP = 4;

template <typename T>
__global__ void decode_ring_kernel(Plan p, int64_t pos_all, const int64_t* pos_dev,
                                   const T* __restrict__ g, T* __restrict__ gc, void* out) {
    __shared__ float part_sum[RP][128];
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
        // slots of its run of tokens pos-w+1 .. pos-1, stepping the slot without a division
        float acc = 0.0f;
        if (pos >= w) {
            const int64_t n = w - 1, per = (n + RP - 1) / RP;
            const int64_t s0 = pos - w + 1 + part * per, s1 = min64(pos, s0 + per);
            int slot = s0 < s1 ? (int)(s0 % R) : 0;
#pragma unroll 4
            for (int64_t s = s0; s < s1; ++s) {
                acc += log_sigmoid<false>(ld(gu + (int64_t)slot * p.D));
                slot = slot + 1 == (int)R ? 0 : slot + 1;
            }
        }
        part_sum[part][f] = acc;
        __syncthreads();
        if (part == 0) {
            float tot = 0.0f;
            if (pos >= w) {
#pragma unroll
                for (int k = 0; k < RP; ++k) tot += part_sum[k][f];
                tot += log_sigmoid<false>(ld(&gnew));
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
    float s = 0.0f;
    for (int64_t j = j0; j < j1; ++j) s += kk[(b * p.L + j) * HD + col];
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
    for (int64_t j = j1 - 1; j >= j0; --j) {
        if (j <= p.L - 1 - p.w) run += x[j * HD];
        x[j * HD] = run;
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
    const unsigned grid = (unsigned)(p.B * p.Hkv), block = (unsigned)(RP * p.D);
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
