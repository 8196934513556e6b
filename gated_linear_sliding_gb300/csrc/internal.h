// Internal host-side interface between the C-ABI entry points and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "lizard.h"

namespace lz {

constexpr int kChunk = 64;            // GLA chunk (tokens); segments are whole chunks
constexpr size_t kHeaderBytes = 256;  // device status word and padding
constexpr int kTargetUnits = 304;     // 2 x 152 SMs: (batch, KV head, segment) CTAs wanted

// Segment plan of a forward/backward call.  The sequence of each (batch, KV head)
// unit is cut into P segments of seg_chunks chunks; the segment count never
// exceeds Pmax, which depends on B and Hkv only, so the workspace does not grow
// with L.
struct Plan {
    int64_t B, L, Hq, Hkv, d, D, w, M, G;
    float scale;
    int dtype;
    int64_t nchunks, seg_chunks, seg_len, P, Pmax;
    size_t rec_floats;   // floats per (segment, unit) record: D*d + D + D
    int64_t rec_step;    // boundary records per segment: the segment pass may cut finer
    // Packed sequences (null: a dense batch): device offsets [B+1]; sequence b is rows
    // [cu[b], cu[b+1]) of arrays with T rows in all, and L is the longest sequence.
    const int64_t* cu = nullptr;
    int64_t T = 0;
    int decay = LIZARD_DECAY_DELAYED;  // lizard_decay: which gates weigh a key past the window
};
// Row of sequence b's first token and the sequence's length (dense batch: b L and L).
__host__ __device__ __forceinline__ int64_t seq_row0(const Plan& p, int64_t b) {
    return p.cu != nullptr ? p.cu[b] : b * p.L;
}
__host__ __device__ __forceinline__ int64_t seq_len(const Plan& p, int64_t b) {
    return p.cu != nullptr ? p.cu[b + 1] - p.cu[b] : p.L;
}

bool make_plan(const lizard_dims* dims, Plan* p);
// Host-side checks shared by every forward entry point (sizes, pointers, alignment, pairs of
// optional outputs, compiled shapes), in this order; fills *p.  Nothing is launched.
lizard_status fwd_check(const lizard_dims* dims, Plan* p, const void* q, const void* k,
                        const void* v, const void* g, const void* Wf, const float* sinks,
                        const void* y, const float* lse, const float* S_out, const float* z_out,
                        const void* kcache_out, const void* vcache_out);
// LIZARD_OK on an sm_103 device, LIZARD_ERR_UNSUPPORTED on another, LIZARD_ERR_CUDA if the
// query fails.
lizard_status device_status();
// Boundary-state records (each rec_floats floats per unit) the forward's launch uses.
// The forward's walk: the tensor-core one on its shapes, except a masked-reading call that
// returns the final state (state_out), which takes the SIMT walk.
bool fwd_uses_tc(const Plan& p, bool state_out);
size_t fwd_records_used(const Plan& p, bool tc);
struct FwdArgs;
// The forward's kernels (tensor-core or SIMT path, then the ring caches) on stream s.
cudaError_t fwd_launch(const Plan& p, const FwdArgs& a, cudaStream_t s);
// Re-cut the segments for a kernel that wants about `target` (unit, segment) CTAs;
// never more than Pmax segments, so the workspace size stays valid.
void plan_segments(Plan* p, int64_t target);
// Re-cut the segments of a kernel that runs one CTA per (unit, segment) on `slots` resident
// CTAs: the segment count (at most Pmax) that minimises waves x segment length.
void plan_segments_waves(Plan* p, int64_t slots);
size_t fwd_workspace_bytes(const Plan& p);

struct FwdArgs {
    const void *q, *k, *v, *g, *Wf;
    const float* sinks;
    void* y;
    float* lse;
    float *S_out, *z_out;
    void *kcache_out, *vcache_out;
    float* seg;   // (Pmax, B*Hkv, rec_floats) segment records
    void* header;
    cudaEvent_t ev_before, ev_after;  // optional: bracket the dominant kernel
    // MASKED and LAGGED readings: reading_scratch_bytes(p) bytes, 256-byte aligned, that
    // fwd_launch fills (the moved gates, or the keys' log gate products)
    void* rscratch = nullptr;
    // MASKED reading: [rows, Hkv, D] log of the product of the w gates after each key (the
    // SIMT walks scale the key's phi by its exponential as it enters the state); else null
    const float* kdec = nullptr;
};

// Reading scratch of a forward (0 for DELAYED): LAGGED moves the gate logits w tokens later
// (one dtype value per gate element), MASKED keeps the keys' log gate products (one fp32).
size_t reading_scratch_bytes(const Plan& p);
// g' = g moved w tokens later in each sequence (rows before w: an open gate, which only
// decays the empty state); out has the layout of g.
cudaError_t launch_gate_lag(const Plan& p, const void* g, void* out, cudaStream_t s);
// kd[j] = sum_{s=j+1..min(j+w, len-1)} log sigmoid(g_s) per (row, KV head, feature).
cudaError_t launch_key_decay(const Plan& p, const void* g, float* kd, cudaStream_t s);
// Gate ring of a prefill: the last min(L, w) tokens' gate rows to slot t mod (w+1).
cudaError_t launch_gate_ring_fill(const Plan& p, const void* g, void* gc, cudaStream_t s);
// Reverse cumulative sum over the rows of each (batch, KV head, feature) column of the
// MASKED backward's key-side gate terms, in place; rows past L - 1 - w (keys that never
// enter the state, not written by the walk) count as zero.  kt: key_suffix_scratch_floats(p)
// floats of chunk totals.
size_t key_suffix_scratch_floats(const Plan& p);
cudaError_t launch_key_suffix(const Plan& p, float* kk, float* kt, cudaStream_t s);

cudaError_t launch_fwd_simt(const Plan& p, const FwdArgs& a, cudaStream_t s);
// Segment-start states only (segment pass + scan into a.seg), for the backward.
cudaError_t launch_fwd_states(const Plan& p, const FwdArgs& a, cudaStream_t s);
// fp32 exclusive scan over the segment records (in place).  dependent: launched to start while
// the kernel before it (the one writing the records) finishes.
cudaError_t launch_seg_scan(const Plan& p, float* seg, cudaStream_t s, bool dependent = false);
bool fwd_tc_supported(const Plan& p);
cudaError_t launch_fwd_tc(const Plan& p, const FwdArgs& a, cudaStream_t s);
// Exact SIMT walk of the segments the tensor-core main walk handed over at a strongly closed
// step (bf16, d = D = 128; p is the tensor-core plan).  Segments not handed over return at once.
cudaError_t launch_fwd_tail(const Plan& p, const FwdArgs& a, cudaStream_t s);
// Segment-start states only (tensor-core segment pass + scan into a.seg), for the backward.
// The segmentation the tensor-core forward runs with (fewest segment-waves on 152 SMs).
void fwd_tc_plan(Plan* p);
cudaError_t launch_fwd_states_tc(const Plan& p, const FwdArgs& a, cudaStream_t s);
cudaError_t launch_ring_fill(const Plan& p, const void* k, const void* v, void* kc, void* vc,
                             cudaStream_t s);

struct DecodeArgs {
    int64_t pos;
    const int64_t* pos_dev;  // per-sequence positions [B] on the device, or null (use pos)
    const void *q, *k, *v, *g, *Wf;
    const float* sinks;
    void* y;
    float *S, *z;
    void *kc, *vc;
    void* header;
    void* gc = nullptr;           // gate-logit ring (MASKED and LAGGED readings)
    const float* kdec = nullptr;  // MASKED: log factor of the admitted key [B, Hkv, D]
};
// Bytes after the status word of a decode workspace (the reading's per-step values).
size_t decode_scratch_bytes(const Plan& p);
// The decode step; for MASKED and LAGGED first the gate-ring step (the step's decay gates
// or the admitted key's factors into the workspace after the status word, the new gate row
// into the ring).
cudaError_t launch_decode(const Plan& p, const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_ring(const Plan& p, const DecodeArgs& a, void* out, cudaStream_t s);

struct BwdArgs {
    const void *q, *k, *v, *g, *Wf;
    const float* sinks;
    const void* y;
    const float* lse;
    const void* dy;
    void *dq, *dk, *dv, *dg;
    float *dWf, *dsinks;
    void* ws;
    size_t ws_bytes;
    cudaEvent_t ev_before, ev_after;
    int win_tc;  // window parts of dq, dk, dv on the tensor cores (set by launch_bwd)
    // set by launch_bwd for the readings: the gate row whose adjoint dg row j takes (LAGGED:
    // j + w), the keys' log gate products and their gate terms (MASKED)
    int64_t glag = 0;
    const float* kdec = nullptr;
    float* kkey = nullptr;
};
size_t bwd_workspace_bytes(const Plan& p);
bool bwd_win_tc_supported(const Plan& p);
bool bwd_rev_local_tc_supported(const Plan& p);
// Reverse-direction walk of the backward on the tensor cores (state parts of dk, dv,
// phi(k')-side of dB with its reverse cumulative sum, dWf and segment totals).
// Segments whose flag is set (flags[seg * B * Hkv + unit] != 0) are left to the SIMT walks.
cudaError_t launch_bwd_rwalk_tc(const Plan& p, const BwdArgs& a, float* wsf, size_t o_rows,
                                size_t o_rev, size_t o_dB, size_t o_dW, size_t o_tot,
                                const int* flags, cudaStream_t s);
// Forward-direction walk of the backward on the tensor cores (state part of dq, phi(q)-side of
// dB, dWf and dt partials); offsets are in floats from the workspace start.
cudaError_t launch_bwd_fwalk_tc(const Plan& p, const BwdArgs& a, float* wsf, size_t o_rows,
                                size_t o_fwd, size_t o_dB, size_t o_dW, size_t o_dt,
                                const int* flags, cudaStream_t s);
// Reverse segment pass on the tensor cores: each segment's contribution to the state adjoint
// at its start (records as the forward's) into rev_rec.
cudaError_t launch_bwd_rev_local_tc(const Plan& p, const BwdArgs& a, const float* rows,
                                    float* rev_rec, cudaStream_t s);
// Window parts of the gradients on the tensor cores: dk, dv (keys) or dq; `rows` is the
// per-row table [e^{-lse}; dy . y].
cudaError_t launch_bwd_win_tc(const Plan& p, const BwdArgs& a, const float* rows, bool keys,
                              cudaStream_t s);
cudaError_t launch_bwd(const Plan& p, const BwdArgs& a, cudaStream_t s);

// The projections in front of the mixer (tcgen05 GEMMs).  proj_supported: bf16, dm a multiple
// of 64, each of Hq d, Hkv d, Hkv D a multiple of 128; *bn is the output tile width.
bool proj_supported(const Plan& p, int64_t dm, int* bn);
cudaError_t launch_proj_fwd(const Plan& p, int64_t dm, const void* x, const void* W, void* q,
                            void* k, void* v, void* g, void* hdr, cudaStream_t s);
cudaError_t launch_proj_bwd(const Plan& p, int64_t dm, const void* x, const void* W,
                            const void* dq, const void* dk, const void* dv, const void* dg,
                            void* dx, float* dW, void* hdr, cudaStream_t s);

// Device address of the status header of lizard_attn_fwd_noalloc's fixed scratch on the
// current device (looked up once per device).
cudaError_t noalloc_header(void** out);

}  // namespace lz
