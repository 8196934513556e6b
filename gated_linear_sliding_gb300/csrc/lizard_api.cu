// C-ABI entry points of the Lizard token-mixer library: argument validation,
// segment planning, workspace sizes and kernel dispatch.  Every check runs on the
// host before any launch; there is no CPU fallback.
#include <algorithm>
#include <vector>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"

namespace lz {

bool make_plan(const lizard_dims* dims, Plan* p) {
    if (dims == nullptr) return false;
    const lizard_dims& d = *dims;
    if (d.B < 1 || d.L < 1 || d.Hq < 1 || d.Hkv < 1 || d.Hq % d.Hkv != 0) return false;
    if (d.w < 1 || d.M < 0 || d.M > 64) return false;
    if (d.D < 2 || d.D % 2 != 0 || d.d < 1) return false;
    if (!(d.chunk == 0 || d.chunk == kChunk)) return false;
    if (!(d.dtype == LIZARD_F32 || d.dtype == LIZARD_BF16)) return false;
    if (!(d.scale >= 0.0f) || !isfinite(d.scale)) return false;
    if (d.decay < LIZARD_DECAY_DELAYED || d.decay > LIZARD_DECAY_LAGGED) return false;
    p->B = d.B;
    p->L = d.L;
    p->Hq = d.Hq;
    p->Hkv = d.Hkv;
    p->d = d.d;
    p->D = d.D;
    p->w = d.w;
    p->M = d.M;
    p->G = d.Hq / d.Hkv;
    p->scale = d.scale > 0.0f ? d.scale : 1.0f / sqrtf((float)d.d);
    p->dtype = d.dtype;
    p->decay = d.decay;
    const int64_t U = d.B * d.Hkv;
    p->nchunks = (d.L + kChunk - 1) / kChunk;
    int64_t pmax = (2 * kTargetUnits + U - 1) / U;
    if (pmax < 1) pmax = 1;
    if (pmax > 64) pmax = 64;
    p->Pmax = pmax;
    p->rec_floats = (size_t)(d.D * d.d + 2 * d.D);
    p->rec_step = 1;
    plan_segments(p, kTargetUnits);
    return true;
}

void plan_segments_waves(Plan* p, int64_t slots) {
    const int64_t U = p->B * p->Hkv;
    int64_t best_cost = -1, best = 1;
    for (int64_t want = 1; want <= p->Pmax; ++want) {
        const int64_t sc = (p->nchunks + want - 1) / want;
        const int64_t P = (p->nchunks + sc - 1) / sc;
        const int64_t cost = ((U * P + slots - 1) / slots) * sc;
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = want;
        }
    }
    p->seg_chunks = (p->nchunks + best - 1) / best;
    p->seg_len = p->seg_chunks * kChunk;
    p->P = (p->nchunks + p->seg_chunks - 1) / p->seg_chunks;
}

void plan_segments(Plan* p, int64_t target) {
    const int64_t U = p->B * p->Hkv;
    int64_t want = (target + U - 1) / U;
    if (want < 1) want = 1;
    if (want > p->Pmax) want = p->Pmax;
    p->seg_chunks = (p->nchunks + want - 1) / want;
    p->seg_len = p->seg_chunks * kChunk;
    p->P = (p->nchunks + p->seg_chunks - 1) / p->seg_chunks;
}

static bool shapes_compiled(const Plan& p) {
    return (p.d == 64 || p.d == 128) && (p.D == 64 || p.D == 128) && p.B * p.Hkv <= 65535 &&
           p.B * p.Hq <= (int64_t)1 << 30;
}

static size_t fwd_base_bytes(const Plan& p) {
    return kHeaderBytes + sizeof(float) * (size_t)p.Pmax * (size_t)(p.B * p.Hkv) * p.rec_floats;
}

static size_t al256(size_t n) { return (n + 255) & ~(size_t)255; }

// The header and the records, then (MASKED and LAGGED readings) the reading's scratch.
size_t fwd_workspace_bytes(const Plan& p) {
    const size_t r = reading_scratch_bytes(p);
    return r == 0 ? fwd_base_bytes(p) : al256(fwd_base_bytes(p)) + r;
}

static void* fwd_reading_scratch(const Plan& p, void* workspace) {
    if (reading_scratch_bytes(p) == 0) return nullptr;
    return (char*)workspace + al256(fwd_base_bytes(p));
}

static bool aligned16(const void* ptr) { return ((uintptr_t)ptr & 15u) == 0; }

lizard_status fwd_check(const lizard_dims* dims, Plan* p, const void* q, const void* k,
                        const void* v, const void* g, const void* Wf, const float* sinks,
                        const void* y, const float* lse, const float* S_out, const float* z_out,
                        const void* kcache_out, const void* vcache_out) {
    if (!make_plan(dims, p)) return LIZARD_ERR_INVALID_ARG;
    if (!q || !k || !v || !g || !Wf || !y || (p->M > 0 && !sinks)) return LIZARD_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, g, Wf, sinks, y, lse, S_out, z_out, kcache_out, vcache_out};
    for (const void* ptr : ptrs)
        if (ptr && !aligned16(ptr)) return LIZARD_ERR_INVALID_ARG;
    if ((S_out == nullptr) != (z_out == nullptr)) return LIZARD_ERR_INVALID_ARG;
    if ((kcache_out == nullptr) != (vcache_out == nullptr)) return LIZARD_ERR_INVALID_ARG;
    if (!shapes_compiled(*p)) return LIZARD_ERR_UNSUPPORTED;
    return LIZARD_OK;
}

bool fwd_uses_tc(const Plan& p, bool state_out) {
    // the masked reading scales each feature row of the state by its keys' gate products, so
    // the final state spans a wide range (max entry ~40x the RMS on the LLaMA-shaped layer);
    // the tensor-core walk's bf16 update operands keep every row's relative error but not
    // the error against the state's RMS, so a masked call returning the state takes the fp32
    // SIMT walk
    return fwd_tc_supported(p) && !(p.decay == LIZARD_DECAY_MASKED && state_out);
}

size_t fwd_records_used(const Plan& p, bool tc) {
    if (tc) {
        Plan pl = p;
        fwd_tc_plan(&pl);
        // every CTA of the tensor-core walk marks its record slot (hand-off to the tail walk)
        return pl.P > 1 ? (size_t)(pl.rec_step * (pl.P - 1) + 1) : 1;
    }
    return p.P > 1 ? (size_t)p.P : 0;
}

cudaError_t fwd_launch(const Plan& p, const FwdArgs& a, cudaStream_t s) {
    // the readings first fill their scratch: the lagged one runs every kernel on the gates
    // moved w tokens later, the masked one gives the SIMT walks the keys' log gate products
    FwdArgs b = a;
    cudaError_t e = cudaSuccess;
    if (p.decay != LIZARD_DECAY_DELAYED) {
        if (a.rscratch == nullptr) return cudaErrorInvalidValue;
        if (p.decay == LIZARD_DECAY_LAGGED) {
            e = launch_gate_lag(p, a.g, a.rscratch, s);
            b.g = a.rscratch;
        } else {
            e = launch_key_decay(p, a.g, (float*)a.rscratch, s);
            b.kdec = (const float*)a.rscratch;
        }
        if (e != cudaSuccess) return e;
    }
    e = fwd_uses_tc(p, a.S_out != nullptr || a.z_out != nullptr) ? launch_fwd_tc(p, b, s)
                                                                 : launch_fwd_simt(p, b, s);
    if (e == cudaSuccess && a.kcache_out != nullptr)
        e = launch_ring_fill(p, a.k, a.v, a.kcache_out, a.vcache_out, s);
    return e;
}

// 1 if the current device is sm_103, 0 if not, -1 if the query failed.
static int device_ok() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    static int cache[64];  // 0 unknown, 1 ok, 2 not ok
    if (dev >= 0 && dev < 64 && cache[dev] != 0) return cache[dev] == 1 ? 1 : 0;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return -1;
    const int ok = (major == 10 && minor == 3) ? 1 : 0;
    if (dev >= 0 && dev < 64) cache[dev] = ok ? 1 : 2;
    return ok;
}

lizard_status device_status() {
    const int ok = device_ok();
    if (ok < 0) {
        cudaGetLastError();
        return LIZARD_ERR_CUDA;
    }
    return ok ? LIZARD_OK : LIZARD_ERR_UNSUPPORTED;
}

static cudaEvent_t g_ev_before = nullptr, g_ev_after = nullptr;

static lizard_status from_cuda(cudaError_t e) { return e == cudaSuccess ? LIZARD_OK : LIZARD_ERR_CUDA; }

}  // namespace lz

using namespace lz;

extern "C" {

size_t lizard_attn_fwd_workspace(const lizard_dims* dims) {
    Plan p;
    if (!make_plan(dims, &p)) return 0;
    return fwd_workspace_bytes(p);
}

int lizard_attn_fwd_kernel(const lizard_dims* dims) {
    Plan p;
    if (!make_plan(dims, &p)) return -1;
    return fwd_tc_supported(p) ? 1 : 0;
}

lizard_status lizard_workspace_init(void* workspace, size_t ws_bytes, void* stream) {
    if (workspace == nullptr || !aligned16(workspace)) return LIZARD_ERR_INVALID_ARG;
    if (ws_bytes < kHeaderBytes) return LIZARD_ERR_WORKSPACE;
    return from_cuda(cudaMemsetAsync(workspace, 0, kHeaderBytes, (cudaStream_t)stream));
}

lizard_status lizard_attn_fwd(const lizard_dims* dims, const void* q, const void* k,
                              const void* v, const void* g, const void* Wf, const float* sinks,
                              void* y, float* lse, float* S_out, float* z_out, void* kcache_out,
                              void* vcache_out, void* workspace, size_t ws_bytes, void* stream) {
    Plan p;
    lizard_status st = fwd_check(dims, &p, q, k, v, g, Wf, sinks, y, lse, S_out, z_out,
                                 kcache_out, vcache_out);
    if (st != LIZARD_OK) return st;
    if (workspace != nullptr && !aligned16(workspace)) return LIZARD_ERR_INVALID_ARG;
    if (workspace == nullptr || ws_bytes < fwd_workspace_bytes(p)) return LIZARD_ERR_WORKSPACE;
    st = device_status();
    if (st != LIZARD_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    FwdArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.Wf = Wf;
    a.sinks = sinks;
    a.y = y;
    a.lse = lse;
    a.S_out = S_out;
    a.z_out = z_out;
    a.kcache_out = kcache_out;
    a.vcache_out = vcache_out;
    a.header = workspace;
    a.seg = (float*)((char*)workspace + kHeaderBytes);
    a.ev_before = g_ev_before;
    a.ev_after = g_ev_after;
    a.rscratch = fwd_reading_scratch(p, workspace);
    return from_cuda(fwd_launch(p, a, s));
}

}  // extern "C"

namespace lz {

static bool packed_offsets_ok(const lizard_dims* dims, const int64_t* cu) {
    if (dims == nullptr || cu == nullptr || dims->B < 1 || dims->L < 0) return false;
    const int64_t nseq = dims->B, T = dims->L;
    if (cu[0] != 0 || cu[nseq] != T) return false;
    for (int64_t i = 0; i < nseq; ++i)
        if (cu[i + 1] < cu[i]) return false;
    return true;
}

// Plan of one launch over all sequences of a packed batch (tensor-core path): sequence b is
// batch b of a plan whose L is the longest sequence.  Segments have one length for all, about
// a quarter of one SM's share of the batch's tokens (whole 64-token chunks), so that CTAs of
// every length even out over the SMs; a sequence's segments past its end walk nothing.  One
// record per (sequence x KV head, segment).  False when the batch is empty or the shapes take
// the SIMT path.
static bool packed_plan(const lizard_dims* dims, const int64_t* cu, Plan* p) {
    const int64_t nseq = dims->B, T = dims->L;
    int64_t lmax = 0;
    for (int64_t i = 0; i < nseq; ++i) lmax = std::max<int64_t>(lmax, cu[i + 1] - cu[i]);
    if (lmax < 1) return false;
    lizard_dims dv = *dims;
    dv.B = nseq;
    dv.L = lmax;
    if (!make_plan(&dv, p)) return false;
    p->T = T;
    // (a masked batch runs sequence by sequence: each call picks its walk, see fwd_uses_tc, by whether it returns the state)
    if (!fwd_tc_supported(*p) || p->decay == LIZARD_DECAY_MASKED) return false;
    const int64_t share = (T * p->Hkv + 151) / 152;
    int64_t sc = (share / 4 + kChunk - 1) / kChunk;
    sc = std::max<int64_t>(1, std::min<int64_t>(sc, p->nchunks));
    p->seg_chunks = sc;
    p->seg_len = sc * kChunk;
    p->P = (p->nchunks + sc - 1) / sc;
    p->Pmax = p->P;
    p->rec_step = 1;
    return true;
}

// Records, then the sequence offsets (copied to the device for the kernels).
static size_t packed_ws_bytes(const Plan& p) {
    return fwd_workspace_bytes(p) + (size_t)(p.B + 1) * sizeof(int64_t);
}

}  // namespace lz

extern "C" {

size_t lizard_attn_fwd_varlen_workspace(const lizard_dims* dims, const int64_t* cu_seqlens) {
    if (!packed_offsets_ok(dims, cu_seqlens)) return 0;
    Plan p;
    if (packed_plan(dims, cu_seqlens, &p)) return packed_ws_bytes(p);
    lizard_dims d1 = *dims;  // one sequence after another
    d1.B = 1;
    d1.L = dims->L > 0 ? dims->L : 1;
    return make_plan(&d1, &p) ? fwd_workspace_bytes(p) : 0;
}

lizard_status lizard_attn_fwd_varlen(const lizard_dims* dims, const int64_t* cu_seqlens,
                                     const void* q, const void* k, const void* v, const void* g,
                                     const void* Wf, const float* sinks, void* y, float* lse,
                                     float* S_out, float* z_out, void* kcache_out,
                                     void* vcache_out, void* workspace, size_t ws_bytes,
                                     void* stream) {
    if (!packed_offsets_ok(dims, cu_seqlens)) return LIZARD_ERR_INVALID_ARG;
    const int64_t nseq = dims->B, T = dims->L;
    cudaStream_t s = (cudaStream_t)stream;
    // one launch over every sequence (tensor-core shapes, workspace of
    // lizard_attn_fwd_varlen_workspace); otherwise the sequences run one after another
    Plan pv;
    if (workspace != nullptr && aligned16(workspace) && packed_plan(dims, cu_seqlens, &pv) &&
        ws_bytes >= packed_ws_bytes(pv)) {
        lizard_dims dv = *dims;
        dv.L = pv.L;
        Plan chk;
        lizard_status st = fwd_check(&dv, &chk, q, k, v, g, Wf, sinks, y, lse, S_out, z_out,
                                     kcache_out, vcache_out);
        if (st != LIZARD_OK) return st;
        st = device_status();
        if (st != LIZARD_OK) return st;
        const size_t Sun = (size_t)(dims->Hkv * dims->D * dims->d), zun = (size_t)(dims->Hkv * dims->D),
                     cun = (size_t)(dims->Hkv * (dims->w + 1) * dims->d) *
                           (dims->dtype == LIZARD_F32 ? 4 : 2);
        cudaError_t e = cudaSuccess;
        for (int64_t i = 0; i < nseq && e == cudaSuccess; ++i) {
            if (cu_seqlens[i + 1] > cu_seqlens[i]) continue;
            // an empty sequence: zero state, empty caches (its segments walk nothing)
            if (S_out) e = cudaMemsetAsync(S_out + (size_t)i * Sun, 0, Sun * sizeof(float), s);
            if (e == cudaSuccess && z_out)
                e = cudaMemsetAsync(z_out + (size_t)i * zun, 0, zun * sizeof(float), s);
            if (e == cudaSuccess && kcache_out)
                e = cudaMemsetAsync((char*)kcache_out + (size_t)i * cun, 0, cun, s);
            if (e == cudaSuccess && vcache_out)
                e = cudaMemsetAsync((char*)vcache_out + (size_t)i * cun, 0, cun, s);
        }
        int64_t* cu_dev = (int64_t*)((char*)workspace + fwd_workspace_bytes(pv));
        if (e == cudaSuccess)  // (from pageable memory: staged before the call returns)
            e = cudaMemcpyAsync(cu_dev, cu_seqlens, (size_t)(nseq + 1) * sizeof(int64_t),
                                cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return from_cuda(e);
        pv.cu = cu_dev;
        FwdArgs a;
        a.q = q;
        a.k = k;
        a.v = v;
        a.g = g;
        a.Wf = Wf;
        a.sinks = sinks;
        a.y = y;
        a.lse = lse;
        a.S_out = S_out;
        a.z_out = z_out;
        a.kcache_out = kcache_out;
        a.vcache_out = vcache_out;
        a.header = workspace;
        a.seg = (float*)((char*)workspace + kHeaderBytes);
        a.ev_before = g_ev_before;
        a.ev_after = g_ev_after;
        a.rscratch = fwd_reading_scratch(pv, workspace);
        return from_cuda(fwd_launch(pv, a, s));
    }
    // every sequence is a B = 1 problem; its workspace does not depend on its length
    lizard_dims d1 = *dims;
    d1.B = 1;
    d1.L = T > 0 ? T : 1;
    Plan p;
    if (!make_plan(&d1, &p)) return LIZARD_ERR_INVALID_ARG;
    if (workspace == nullptr || ws_bytes < fwd_workspace_bytes(p)) return LIZARD_ERR_WORKSPACE;
    const size_t E = d1.dtype == LIZARD_F32 ? 4 : 2;
    const size_t qrow = (size_t)(d1.Hq * d1.d) * E, krow = (size_t)(d1.Hkv * d1.d) * E,
                 grow = (size_t)(d1.Hkv * d1.D) * E;
    const size_t Sun = (size_t)(d1.Hkv * d1.D * d1.d), zun = (size_t)(d1.Hkv * d1.D),
                 cun = (size_t)(d1.Hkv * (d1.w + 1) * d1.d) * E;
    for (int64_t i = 0; i < nseq; ++i) {
        const int64_t t0 = cu_seqlens[i], n = cu_seqlens[i + 1] - t0;
        float* Si = S_out ? S_out + (size_t)i * Sun : nullptr;
        float* zi = z_out ? z_out + (size_t)i * zun : nullptr;
        char* kci = kcache_out ? (char*)kcache_out + (size_t)i * cun : nullptr;
        char* vci = vcache_out ? (char*)vcache_out + (size_t)i * cun : nullptr;
        if (n == 0) {  // an empty sequence: zero state, empty caches
            cudaError_t e = cudaSuccess;
            if (Si) e = cudaMemsetAsync(Si, 0, Sun * sizeof(float), s);
            if (e == cudaSuccess && zi) e = cudaMemsetAsync(zi, 0, zun * sizeof(float), s);
            if (e == cudaSuccess && kci) e = cudaMemsetAsync(kci, 0, cun, s);
            if (e == cudaSuccess && vci) e = cudaMemsetAsync(vci, 0, cun, s);
            if (e != cudaSuccess) return from_cuda(e);
            continue;
        }
        d1.L = n;
        const lizard_status st = lizard_attn_fwd(
            &d1, (const char*)q + t0 * qrow, (const char*)k + t0 * krow,
            (const char*)v + t0 * krow, (const char*)g + t0 * grow, Wf, sinks,
            (char*)y + t0 * qrow, lse ? lse + t0 * d1.Hq : nullptr, Si, zi, kci, vci, workspace,
            ws_bytes, stream);
        if (st != LIZARD_OK) return st;
    }
    return LIZARD_OK;
}

size_t lizard_attn_bwd_workspace(const lizard_dims* dims) {
    Plan p;
    if (!make_plan(dims, &p)) return 0;
    return bwd_workspace_bytes(p);
}

lizard_status lizard_attn_bwd(const lizard_dims* dims, const void* q, const void* k,
                              const void* v, const void* g, const void* Wf, const float* sinks,
                              const void* y, const float* lse, const void* dy, void* dq, void* dk,
                              void* dv, void* dg, float* dWf, float* dsinks, void* workspace,
                              size_t ws_bytes, void* stream) {
    Plan p;
    if (!make_plan(dims, &p)) return LIZARD_ERR_INVALID_ARG;
    const void* req[] = {q, k, v, g, Wf, y, lse, dy, dq, dk, dv, dg, dWf};
    for (const void* ptr : req)
        if (ptr == nullptr || !aligned16(ptr)) return LIZARD_ERR_INVALID_ARG;
    if (p.M > 0 && (!sinks || !dsinks || !aligned16(sinks) || !aligned16(dsinks)))
        return LIZARD_ERR_INVALID_ARG;
    if (!shapes_compiled(p)) return LIZARD_ERR_UNSUPPORTED;
    if (workspace == nullptr || !aligned16(workspace) || ws_bytes < bwd_workspace_bytes(p))
        return LIZARD_ERR_WORKSPACE;
    lizard_status st = device_status();
    if (st != LIZARD_OK) return st;
    BwdArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.Wf = Wf;
    a.sinks = sinks;
    a.y = y;
    a.lse = lse;
    a.dy = dy;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.dg = dg;
    a.dWf = dWf;
    a.dsinks = dsinks;
    a.ws = workspace;
    a.ws_bytes = ws_bytes;
    a.ev_before = g_ev_before;
    a.ev_after = g_ev_after;
    return from_cuda(launch_bwd(p, a, (cudaStream_t)stream));
}

// Packed-batch backward: dst = src (first sequence) or dst += src (the others), fixed order.
__global__ void add_or_copy(float* dst, const float* src, size_t n, int first) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) dst[i] = first ? src[i] : dst[i] + src[i];
}

static bool varlen_offsets_ok(const lizard_dims* dims, const int64_t* cu) {
    if (dims == nullptr || cu == nullptr || dims->B < 1 || dims->L < 0) return false;
    if (cu[0] != 0 || cu[dims->B] != dims->L) return false;
    for (int64_t i = 0; i < dims->B; ++i)
        if (cu[i + 1] < cu[i]) return false;
    return true;
}

// The largest B = 1 backward workspace over the sequences, 256-byte aligned, then the
// per-sequence dWf and dsinks.
static size_t bwd_varlen_main_bytes(const lizard_dims* dims, const int64_t* cu) {
    lizard_dims d1 = *dims;
    d1.B = 1;
    d1.L = 1;
    for (int64_t i = 0; i < dims->B; ++i) d1.L = cu[i + 1] - cu[i] > d1.L ? cu[i + 1] - cu[i] : d1.L;
    Plan p;
    if (!make_plan(&d1, &p)) return 0;
    return (bwd_workspace_bytes(p) + 255) & ~(size_t)255;
}

}  // extern "C"

namespace lz {

// The packed backward runs its sequences as independent backwards on kBwdLanes streams, forked
// from the caller's stream and joined back before the call returns; each lane has its own
// slice of the workspace (its own status word) and its own dWf, dsinks partials.
constexpr int kBwdLanes = 4;

struct LanePool {
    int dev = -1;
    cudaStream_t s[kBwdLanes];
    cudaEvent_t done[kBwdLanes], fork;
};
static LanePool g_lanes;

// The lanes' streams and events, made once for the first device that asks (null on another).
static LanePool* lane_pool() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    if (g_lanes.dev == dev) return &g_lanes;
    if (g_lanes.dev != -1) return nullptr;
    for (int k = 0; k < kBwdLanes; ++k) {
        if (cudaStreamCreateWithFlags(&g_lanes.s[k], cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&g_lanes.done[k], cudaEventDisableTiming) != cudaSuccess)
            return nullptr;
    }
    if (cudaEventCreateWithFlags(&g_lanes.fork, cudaEventDisableTiming) != cudaSuccess)
        return nullptr;
    g_lanes.dev = dev;
    return &g_lanes;
}

static size_t round256(size_t n) { return (n + 255) & ~(size_t)255; }

// dst[i] = sum over the lanes in `mask`, lane 0 first, of src[k stride + i].
__global__ void sum_lanes(float* dst, const float* src, size_t n, size_t stride, unsigned mask) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float acc = 0.0f;
    bool first = true;
    for (int k = 0; k < kBwdLanes; ++k) {
        if (!((mask >> k) & 1u)) continue;
        acc = first ? src[(size_t)k * stride + i] : acc + src[(size_t)k * stride + i];
        first = false;
    }
    dst[i] = acc;
}

// The first error a lane recorded reaches the caller's status word; lane words are cleared.
__global__ void merge_lane_status(WsHeader* head, char* ws, size_t lane_bytes) {
    if (threadIdx.x != 0) return;
    for (int k = 1; k < kBwdLanes; ++k) {
        WsHeader* h = (WsHeader*)(ws + (size_t)k * lane_bytes);
        if (h->status != 0u && head->status == 0u) {
            head->status = h->status;
            head->where = h->where;
        }
        h->status = 0u;
        h->where = 0u;
    }
}

}  // namespace lz

extern "C" {

size_t lizard_attn_bwd_varlen_workspace(const lizard_dims* dims, const int64_t* cu_seqlens) {
    if (!varlen_offsets_ok(dims, cu_seqlens)) return 0;
    const size_t main = bwd_varlen_main_bytes(dims, cu_seqlens);
    if (main == 0) return 0;
    const size_t nW = (size_t)(dims->Hkv * dims->d * (dims->D / 2)), nt = (size_t)(dims->Hq * dims->M);
    // per lane: a backward's workspace, the dWf and dsinks of one sequence, the lane's sums
    return (size_t)kBwdLanes * (main + 2 * round256(nW * 4) + 2 * round256(nt * 4));
}

lizard_status lizard_attn_bwd_varlen(const lizard_dims* dims, const int64_t* cu_seqlens,
                                     const void* q, const void* k, const void* v, const void* g,
                                     const void* Wf, const float* sinks, const void* y,
                                     const float* lse, const void* dy, void* dq, void* dk,
                                     void* dv, void* dg, float* dWf, float* dsinks,
                                     void* workspace, size_t ws_bytes, void* stream) {
    if (!varlen_offsets_ok(dims, cu_seqlens)) return LIZARD_ERR_INVALID_ARG;
    const size_t need_lanes = lizard_attn_bwd_varlen_workspace(dims, cu_seqlens);
    if (need_lanes == 0) return LIZARD_ERR_INVALID_ARG;
    const size_t main = bwd_varlen_main_bytes(dims, cu_seqlens);
    const size_t nW = (size_t)(dims->Hkv * dims->d * (dims->D / 2)), nt = (size_t)(dims->Hq * dims->M);
    const size_t rW = round256(nW * 4), rt = round256(nt * 4);
    // one backward at a time needs a single lane's share
    if (workspace == nullptr || ws_bytes < main + rW + rt) return LIZARD_ERR_WORKSPACE;
    if (dWf == nullptr || (dims->M > 0 && dsinks == nullptr)) return LIZARD_ERR_INVALID_ARG;
    LanePool* pool = ws_bytes >= need_lanes && dims->B > 1 ? lane_pool() : nullptr;
    if (pool != nullptr) {
        cudaStream_t s = (cudaStream_t)stream;
        char* ws = (char*)workspace;
        char* temps = ws + (size_t)kBwdLanes * main;   // [lane] dWf, then [lane] dsinks of one sequence
        char* sums = temps + (size_t)kBwdLanes * (rW + rt);  // the lanes' running sums, same layout
        auto tW = [&](int ln) { return (float*)(temps + (size_t)ln * rW); };
        auto tt = [&](int ln) { return (float*)(temps + (size_t)kBwdLanes * rW + (size_t)ln * rt); };
        auto aW = [&](int ln) { return (float*)(sums + (size_t)ln * rW); };
        auto at = [&](int ln) { return (float*)(sums + (size_t)kBwdLanes * rW + (size_t)ln * rt); };
        // longest sequences first, each to the lane with the fewest tokens so far (ties: lower
        // lane); each lane then runs its sequences in index order
        const int64_t nseq = dims->B;
        std::vector<int64_t> order(nseq);
        for (int64_t i = 0; i < nseq; ++i) order[i] = i;
        std::stable_sort(order.begin(), order.end(), [&](int64_t x, int64_t y) {
            return cu_seqlens[x + 1] - cu_seqlens[x] > cu_seqlens[y + 1] - cu_seqlens[y];
        });
        std::vector<int> lane_of(nseq, 0);
        int64_t load[kBwdLanes] = {};
        for (int64_t i : order) {
            int best = 0;
            for (int ln = 1; ln < kBwdLanes; ++ln)
                if (load[ln] < load[best]) best = ln;
            lane_of[i] = best;
            load[best] += cu_seqlens[i + 1] - cu_seqlens[i];
        }
        cudaError_t e = cudaSuccess;
        for (int ln = 1; ln < kBwdLanes && e == cudaSuccess; ++ln)  // the lanes' status words
            e = cudaMemsetAsync(ws + (size_t)ln * main, 0, kHeaderBytes, s);
        if (e == cudaSuccess) e = cudaEventRecord(pool->fork, s);
        for (int ln = 0; ln < kBwdLanes && e == cudaSuccess; ++ln)
            e = cudaStreamWaitEvent(pool->s[ln], pool->fork, 0);
        if (e != cudaSuccess) return from_cuda(e);
        lizard_dims d1 = *dims;
        d1.B = 1;
        const size_t E = d1.dtype == LIZARD_F32 ? 4 : 2;
        const size_t qrow = (size_t)(d1.Hq * d1.d) * E, krow = (size_t)(d1.Hkv * d1.d) * E,
                     grow = (size_t)(d1.Hkv * d1.D) * E;
        unsigned used = 0u;
        lizard_status st = LIZARD_OK;
        for (int64_t i = 0; i < nseq && st == LIZARD_OK; ++i) {
            const int64_t t0 = cu_seqlens[i], n = cu_seqlens[i + 1] - t0;
            if (n == 0) continue;  // no tokens: no gradient slice, nothing to add
            const int ln = lane_of[i];
            cudaStream_t ls = pool->s[ln];
            d1.L = n;
            st = lizard_attn_bwd(
                &d1, (const char*)q + t0 * qrow, (const char*)k + t0 * krow,
                (const char*)v + t0 * krow, (const char*)g + t0 * grow, Wf, sinks,
                (const char*)y + t0 * qrow, lse + t0 * d1.Hq, (const char*)dy + t0 * qrow,
                (char*)dq + t0 * qrow, (char*)dk + t0 * krow, (char*)dv + t0 * krow,
                (char*)dg + t0 * grow, tW(ln), dims->M > 0 ? tt(ln) : nullptr,
                ws + (size_t)ln * main, main, ls);
            if (st != LIZARD_OK) break;
            const int first = (used >> ln) & 1u ? 0 : 1;
            add_or_copy<<<(unsigned)((nW + 255) / 256), 256, 0, ls>>>(aW(ln), tW(ln), nW, first);
            if (dims->M > 0)
                add_or_copy<<<(unsigned)((nt + 255) / 256), 256, 0, ls>>>(at(ln), tt(ln), nt, first);
            if (cudaGetLastError() != cudaSuccess) st = LIZARD_ERR_CUDA;
            used |= 1u << ln;
        }
        // every lane joins the caller's stream, whatever happened above
        for (int ln = 0; ln < kBwdLanes; ++ln) {
            if (cudaEventRecord(pool->done[ln], pool->s[ln]) != cudaSuccess ||
                cudaStreamWaitEvent(s, pool->done[ln], 0) != cudaSuccess)
                st = LIZARD_ERR_CUDA;
        }
        if (st != LIZARD_OK) return st;
        if (used == 0u) {  // every sequence is empty: zero parameter gradients
            e = cudaMemsetAsync(dWf, 0, nW * 4, s);
            if (e == cudaSuccess && dims->M > 0) e = cudaMemsetAsync(dsinks, 0, nt * 4, s);
        } else {
            sum_lanes<<<(unsigned)((nW + 255) / 256), 256, 0, s>>>(dWf, aW(0), nW, rW / 4, used);
            if (dims->M > 0)
                sum_lanes<<<(unsigned)((nt + 255) / 256), 256, 0, s>>>(dsinks, at(0), nt, rt / 4, used);
            e = cudaGetLastError();
        }
        if (e == cudaSuccess) {
            merge_lane_status<<<1, 32, 0, s>>>((WsHeader*)ws, ws, main);
            e = cudaGetLastError();
        }
        return from_cuda(e);
    }
    float* tW = (float*)((char*)workspace + main);
    float* tt = (float*)((char*)workspace + main + rW);
    lizard_dims d1 = *dims;
    d1.B = 1;
    const size_t E = d1.dtype == LIZARD_F32 ? 4 : 2;
    const size_t qrow = (size_t)(d1.Hq * d1.d) * E, krow = (size_t)(d1.Hkv * d1.d) * E,
                 grow = (size_t)(d1.Hkv * d1.D) * E;
    cudaStream_t s = (cudaStream_t)stream;
    bool first = true;
    for (int64_t i = 0; i < dims->B; ++i) {
        const int64_t t0 = cu_seqlens[i], n = cu_seqlens[i + 1] - t0;
        if (n == 0) continue;  // no tokens: no gradient slice, nothing to add
        d1.L = n;
        const lizard_status st = lizard_attn_bwd(
            &d1, (const char*)q + t0 * qrow, (const char*)k + t0 * krow,
            (const char*)v + t0 * krow, (const char*)g + t0 * grow, Wf, sinks,
            (const char*)y + t0 * qrow, lse + t0 * d1.Hq, (const char*)dy + t0 * qrow,
            (char*)dq + t0 * qrow, (char*)dk + t0 * krow, (char*)dv + t0 * krow,
            (char*)dg + t0 * grow, tW, dims->M > 0 ? tt : nullptr, workspace, main, stream);
        if (st != LIZARD_OK) return st;
        add_or_copy<<<(unsigned)((nW + 255) / 256), 256, 0, s>>>(dWf, tW, nW, first ? 1 : 0);
        if (dims->M > 0)
            add_or_copy<<<(unsigned)((nt + 255) / 256), 256, 0, s>>>(dsinks, tt, nt, first ? 1 : 0);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return from_cuda(e);
        first = false;
    }
    if (first) {  // every sequence is empty: zero parameter gradients
        cudaError_t e = cudaMemsetAsync(dWf, 0, nW * 4, s);
        if (e == cudaSuccess && dims->M > 0) e = cudaMemsetAsync(dsinks, 0, nt * 4, s);
        if (e != cudaSuccess) return from_cuda(e);
    }
    return LIZARD_OK;
}

size_t lizard_decode_workspace(const lizard_dims* dims) {
    lizard_dims d1 = dims ? *dims : lizard_dims{};
    d1.L = 1;
    Plan p;
    if (!make_plan(&d1, &p)) return 0;
    return kHeaderBytes + decode_scratch_bytes(p);
}

lizard_status lizard_gate_cache_fill(const lizard_dims* dims, const void* g, void* gcache,
                                     void* stream) {
    Plan p;
    if (!make_plan(dims, &p) || g == nullptr || gcache == nullptr || !aligned16(g) ||
        !aligned16(gcache))
        return LIZARD_ERR_INVALID_ARG;
    if (!shapes_compiled(p)) return LIZARD_ERR_UNSUPPORTED;
    const lizard_status st = device_status();
    if (st != LIZARD_OK) return st;
    return from_cuda(launch_gate_ring_fill(p, g, gcache, (cudaStream_t)stream));
}

// Both decode entry points: one position for the batch (pos_dev null) or one per sequence.
static lizard_status decode_step(const lizard_dims* dims, int64_t pos, const int64_t* pos_dev,
                                 const void* q, const void* k, const void* v, const void* g,
                                 const void* Wf, const float* sinks, void* y, float* S, float* z,
                                 void* kcache, void* vcache, void* gcache, void* workspace,
                                 size_t ws_bytes, void* stream) {
    if (dims == nullptr) return LIZARD_ERR_INVALID_ARG;
    lizard_dims d1 = *dims;
    d1.L = 1;
    Plan p;
    if (!make_plan(&d1, &p) || pos < 0) return LIZARD_ERR_INVALID_ARG;
    const void* req[] = {q, k, v, g, Wf, y, S, z, kcache, vcache};
    for (const void* ptr : req)
        if (ptr == nullptr || !aligned16(ptr)) return LIZARD_ERR_INVALID_ARG;
    if (p.M > 0 && (!sinks || !aligned16(sinks))) return LIZARD_ERR_INVALID_ARG;
    // the masked and lagged readings decay or weigh with gates of the window's tokens
    if (p.decay != LIZARD_DECAY_DELAYED && (gcache == nullptr || !aligned16(gcache)))
        return LIZARD_ERR_INVALID_ARG;
    if (!shapes_compiled(p) || p.G > 8 || p.w > 256) return LIZARD_ERR_UNSUPPORTED;
    if (workspace == nullptr || !aligned16(workspace) ||
        ws_bytes < kHeaderBytes + decode_scratch_bytes(p))
        return LIZARD_ERR_WORKSPACE;
    lizard_status st = device_status();
    if (st != LIZARD_OK) return st;
    DecodeArgs a;
    a.pos = pos;
    a.pos_dev = pos_dev;
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.Wf = Wf;
    a.sinks = sinks;
    a.y = y;
    a.S = S;
    a.z = z;
    a.kc = kcache;
    a.vc = vcache;
    a.header = workspace;
    a.gc = p.decay != LIZARD_DECAY_DELAYED ? gcache : nullptr;
    return from_cuda(launch_decode(p, a, (cudaStream_t)stream));
}

lizard_status lizard_decode_step(const lizard_dims* dims, int64_t pos, const void* q,
                                 const void* k, const void* v, const void* g, const void* Wf,
                                 const float* sinks, void* y, float* S, float* z, void* kcache,
                                 void* vcache, void* gcache, void* workspace, size_t ws_bytes,
                                 void* stream) {
    return decode_step(dims, pos, nullptr, q, k, v, g, Wf, sinks, y, S, z, kcache, vcache,
                       gcache, workspace, ws_bytes, stream);
}

lizard_status lizard_decode_step_positions(const lizard_dims* dims, const int64_t* pos,
                                           const void* q, const void* k, const void* v,
                                           const void* g, const void* Wf, const float* sinks,
                                           void* y, float* S, float* z, void* kcache,
                                           void* vcache, void* gcache, void* workspace,
                                           size_t ws_bytes, void* stream) {
    if (pos == nullptr || ((uintptr_t)pos & 7u) != 0) return LIZARD_ERR_INVALID_ARG;
    return decode_step(dims, 0, pos, q, k, v, g, Wf, sinks, y, S, z, kcache, vcache, gcache,
                       workspace, ws_bytes, stream);
}

// Checks shared by the two projection entry points.
static lizard_status proj_check(const lizard_dims* dims, int64_t dmodel, Plan* p,
                                const void* const* ptrs, int n, void* workspace,
                                size_t ws_bytes) {
    if (!make_plan(dims, p) || dmodel < 1) return LIZARD_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i)
        if (ptrs[i] == nullptr || !aligned16(ptrs[i])) return LIZARD_ERR_INVALID_ARG;
    if (workspace != nullptr && !aligned16(workspace)) return LIZARD_ERR_INVALID_ARG;
    int bn = 0;
    if (!proj_supported(*p, dmodel, &bn)) return LIZARD_ERR_UNSUPPORTED;
    if (workspace != nullptr && ws_bytes < kHeaderBytes) return LIZARD_ERR_WORKSPACE;
    return device_status();
}

lizard_status lizard_qkvg_proj(const lizard_dims* dims, int64_t dmodel, const void* x,
                               const void* W, void* q, void* k, void* v, void* g,
                               void* workspace, size_t ws_bytes, void* stream) {
    Plan p;
    const void* ptrs[] = {x, W, q, k, v, g};
    const lizard_status st = proj_check(dims, dmodel, &p, ptrs, 6, workspace, ws_bytes);
    if (st != LIZARD_OK) return st;
    return from_cuda(launch_proj_fwd(p, dmodel, x, W, q, k, v, g, workspace,
                                     (cudaStream_t)stream));
}

lizard_status lizard_qkvg_proj_bwd(const lizard_dims* dims, int64_t dmodel, const void* x,
                                   const void* W, const void* dq, const void* dk,
                                   const void* dv, const void* dg, void* dx, float* dW,
                                   void* workspace, size_t ws_bytes, void* stream) {
    Plan p;
    const void* ptrs[] = {x, W, dq, dk, dv, dg, dx, dW};
    const lizard_status st = proj_check(dims, dmodel, &p, ptrs, 8, workspace, ws_bytes);
    if (st != LIZARD_OK) return st;
    return from_cuda(launch_proj_bwd(p, dmodel, x, W, dq, dk, dv, dg, dx, dW, workspace,
                                     (cudaStream_t)stream));
}

lizard_status lizard_read_device_status(void* workspace, void* stream) {
    if (workspace == nullptr || !aligned16(workspace)) return LIZARD_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaStreamSynchronize(s) != cudaSuccess) return LIZARD_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return LIZARD_ERR_CUDA;
    if (word != 0 && cudaMemset(workspace, 0, kHeaderBytes) != cudaSuccess)
        return LIZARD_ERR_CUDA;
    if (word > (unsigned)LIZARD_ERR_TIMEOUT) return LIZARD_ERR_CUDA;
    return (lizard_status)word;
}

const char* lizard_status_string(lizard_status s) {
    switch (s) {
        case LIZARD_OK: return "ok";
        case LIZARD_ERR_INVALID_ARG: return "invalid argument";
        case LIZARD_ERR_UNSUPPORTED: return "unsupported sizes or device";
        case LIZARD_ERR_WORKSPACE: return "workspace missing or too small";
        case LIZARD_ERR_CUDA: return "CUDA error";
        case LIZARD_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

lizard_status lizard_profile_events(void* before, void* after) {
    if ((before == nullptr) != (after == nullptr)) return LIZARD_ERR_INVALID_ARG;
    g_ev_before = (cudaEvent_t)before;
    g_ev_after = (cudaEvent_t)after;
    return LIZARD_OK;
}

const char* lizard_version(void) { return "lizard-gb300 0.1 (sm_103a)"; }

}  // extern "C"
