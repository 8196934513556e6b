/*
 * lizard.h - C ABI of the GB300 (sm_103a) Lizard hybrid token mixer.
 *
 * The mixer (Lizard summary, gist.science/ko/paper/2507.09025):
 *   sec. 2-A-1  gated linear attention: a data-dependent gate
 *               Gamma_i = sigmoid(g_i) (per token, per feature) decays a
 *               constant-size state S_i updated token by token;
 *   sec. 2-A-2  sliding-window softmax attention whose denominator also holds
 *               learnable meta-memory scalars t_m ("sinks");
 *   sec. 2-C    the non-negative Hedgehog feature map
 *               phi(x) = [softmax(x Wf), softmax(-x Wf)], which lets the gates
 *               move to log space and fold into the query/key sides.
 * Both parts share one normaliser:
 *   y_i = [phi(q_i) S_i + sum_{j in (i-w, i]} e^{s q_i.k_j} v_j]
 *       / [phi(q_i).z_i + sum_{j in (i-w, i]} e^{s q_i.k_j} + sum_m e^{t_m}],
 *   S_i = Gamma_i (.) S_{i-1} + [i >= w] phi(k_{i-w}) v_{i-w}^T,
 *   z_i = Gamma_i (.) z_{i-1} + [i >= w] phi(k_{i-w}),
 * i.e. a key enters the state, undecayed, at the step it leaves the window and
 * is decayed by every later gate.  Query head h uses KV head h / (Hq / Hkv),
 * which owns Wf, the gate logits, S and z.
 *
 * The pages say only that the gate decays a state of the tokens outside the
 * window (sec. 2-A-1), not which gates a key that has left the window has seen.
 * The recurrence above is the default reading; dims.decay selects one of two
 * others, as the gate product that weighs key j <= i - w at query i:
 *   LIZARD_DECAY_DELAYED (0)  prod_{s=j+w+1..i} Gamma_s  (the recurrence above);
 *   LIZARD_DECAY_MASKED  (1)  prod_{s=j+1..i}   Gamma_s  (full gated linear
 *       attention with the window's keys masked out: the key enters the state
 *       already decayed by the w gates it saw inside the window);
 *   LIZARD_DECAY_LAGGED  (2)  prod_{s=j+1..i-w} Gamma_s  (the query reads the
 *       gated state of token i - w: the delayed recurrence run on the gates of
 *       w tokens earlier).
 * All three coincide when every gate is 1.
 *
 * Conventions for every entry point:
 *   - All tensor arguments are DEVICE pointers to contiguous row-major arrays,
 *     16-byte aligned.  The caller allocates and owns every buffer, workspace
 *     included.  The library never allocates, frees or synchronises (except
 *     lizard_read_device_status) and enqueues all work on `stream` (a
 *     cudaStream_t; NULL = legacy default stream).
 *   - Arguments are validated on the host before any launch; on any error the
 *     call returns a status and launches nothing.
 *   - Element type `dtype` (LIZARD_F32 or LIZARD_BF16) applies to q, k, v, g,
 *     Wf, y, the ring caches and the gradients dq, dk, dv, dg.  sinks, S, z,
 *     lse, dWf and dsinks are always fp32.
 *   - Positions are 0-based.  There is no CPU fallback: on a device other than
 *     sm_103 every call returns LIZARD_ERR_UNSUPPORTED.
 *
 * Layouts:
 *   q, y, dy, dq  [B, L, Hq, d]        k, v, dk, dv  [B, L, Hkv, d]
 *   g, dg         [B, L, Hkv, D]       Wf, dWf       [Hkv, d, D/2]
 *   sinks, dsinks [Hq, M] (fp32)       lse           [B, L, Hq] (fp32)
 *   S             [B, Hkv, D, d] fp32  z             [B, Hkv, D] fp32
 *   kcache/vcache [B, Hkv, w+1, d]     token t lives in slot t mod (w+1)
 *   gcache        [B, Hkv, w+1, D]     gate logits, same slots (MASKED/LAGGED decode)
 */
#ifndef LIZARD_H
#define LIZARD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LIZARD_OK = 0,
    LIZARD_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, inconsistent sizes      */
    LIZARD_ERR_UNSUPPORTED = 2,  /* sizes outside the compiled kernels, or not sm_103 */
    LIZARD_ERR_WORKSPACE = 3,    /* workspace NULL or smaller than the query says     */
    LIZARD_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed               */
    LIZARD_ERR_TIMEOUT = 5       /* a bounded device-side wait gave up (device status) */
} lizard_status;

typedef enum { LIZARD_F32 = 0, LIZARD_BF16 = 1 } lizard_dtype;

typedef enum {
    LIZARD_DECAY_DELAYED = 0, /* key enters undecayed as it leaves the window (default) */
    LIZARD_DECAY_MASKED = 1,  /* full gated linear attention, window masked out        */
    LIZARD_DECAY_LAGGED = 2   /* the query reads the gated state of token i - w         */
} lizard_decay;

/* Problem sizes.  d, D in {64, 128}; D is the phi width (Wf is d x D/2);
 * Hq % Hkv == 0; w >= 1 (window of the w most recent tokens, self included);
 * 0 <= M <= 64 sinks per query head; chunk is 0 (default) or 64;
 * scale is the softmax scale applied to q.k, 0 selects 1/sqrt(d);
 * decay is the reading of the gate decay (lizard_decay; 0, the default, in a
 * zero-initialised struct).  How each reading runs:
 *   DELAYED  every path below as described;
 *   LAGGED   the same kernels on the gate logits moved w tokens later (a copy in
 *            the workspace, B L Hkv D elements more than the DELAYED workspace; the
 *            backward moves dg back); decode needs the gate ring (gcache);
 *   MASKED   each entering key's phi scaled by the product of the w gates it saw in the
 *            window (per-token log products in the workspace, B L Hkv D fp32 more): the
 *            forward folds the factor into the keys' decay tables (tensor-core walk, or
 *            the SIMT walk when the call returns the final state, see
 *            lizard_attn_fwd_kernel; a packed batch runs sequence by sequence); the
 *            backward's state walks take the same factor and keep the key-side gate terms
 *            in a second such array; decode needs gcache. */
typedef struct {
    int64_t B, L, Hq, Hkv, d, D, w, M;
    int64_t chunk;
    float scale;
    int32_t dtype; /* lizard_dtype */
    int32_t decay; /* lizard_decay */
} lizard_dims;

/* Bytes of device workspace lizard_attn_fwd needs.  Under the DELAYED reading it
 * depends on B, Hkv, d and D only, never on L (the per-segment boundary states,
 * sec. 2-A-1 constant memory); the MASKED and LAGGED readings add one value per gate
 * element (see lizard_dims).  Returns 0 for invalid dims. */
size_t lizard_attn_fwd_workspace(const lizard_dims* dims);

/* Which forward kernel serves these sizes: 1 = the tensor-core (tcgen05) chunk walk
 * (bf16, d = D = 128, Hq = 4 Hkv, w = 64), 0 = the SIMT walk (fp32 and every other
 * shape), -1 = invalid sizes.  Under the MASKED reading a call that returns the final state
 * (S_out, z_out) takes the SIMT walk even on the tensor-core shapes: that state spans a wide
 * range (each feature row scaled by its keys' gate products), which the tensor-core walk's
 * bf16 update operands do not hold to the bf16 bound against its RMS.  Pure host query. */
int lizard_attn_fwd_kernel(const lizard_dims* dims);

/* Zero the device status word at the head of a workspace (async on stream).
 * Call once after allocating a workspace; kernels only ever set the word. */
lizard_status lizard_workspace_init(void* workspace, size_t ws_bytes, void* stream);

/* Prefill / training forward over L tokens (sec. 2-A-1, 2-A-2, 2-C).
 *   q, k, v, g, Wf, sinks   inputs as laid out above (read only);
 *   y                       output [B, L, Hq, d];
 *   lse                     optional (NULL to skip) [B, L, Hq] fp32: natural log
 *                           of each row's full denominator, kept for the backward;
 *   S_out, z_out            optional final state after token L-1 (decode hand-off);
 *   kcache_out, vcache_out  optional ring caches: the last min(L, w) tokens are
 *                           written to slot t mod (w+1), other slots untouched;
 *   workspace, ws_bytes     >= lizard_attn_fwd_workspace(dims) bytes. */
lizard_status lizard_attn_fwd(const lizard_dims* dims, const void* q, const void* k,
                              const void* v, const void* g, const void* Wf, const float* sinks,
                              void* y, float* lse, float* S_out, float* z_out, void* kcache_out,
                              void* vcache_out, void* workspace, size_t ws_bytes, void* stream);

/* Bytes of device workspace for one launch of lizard_attn_fwd_varlen over all sequences of
 * this packed batch (dims.B sequences, dims.L tokens in all, host offsets cu_seqlens as
 * below): the header, one boundary record of (D d + 2 D) floats per (sequence x KV head,
 * segment) and the B + 1 offsets.  For shapes that run one sequence at a time it is the
 * workspace of a single sequence.  0 for invalid dims or offsets. */
size_t lizard_attn_fwd_varlen_workspace(const lizard_dims* dims, const int64_t* cu_seqlens);

/* The forward over a packed batch of sequences of different lengths (variable-length
 * batching).  dims.B is the number of sequences and dims.L the total number of tokens T;
 * cu_seqlens is a HOST array of B + 1 offsets (cu_seqlens[0] = 0, non-decreasing,
 * cu_seqlens[B] = T): sequence i is tokens [cu_seqlens[i], cu_seqlens[i+1]).
 *   q, y [T, Hq, d]; k, v [T, Hkv, d]; g [T, Hkv, D]; lse (nullable) [T, Hq] fp32; the
 *   packed layouts are those of lizard_attn_fwd with B = 1 and L = T.
 *   S_out, z_out, kcache_out, vcache_out (nullable, in pairs) hold one entry per sequence:
 *   [B, Hkv, D, d], [B, Hkv, D], [B, Hkv, w+1, d]; an empty sequence gets a zero state.
 *   workspace: ws_bytes >= lizard_attn_fwd_varlen_workspace(dims, cu_seqlens) gives one
 *   launch over all sequences; a workspace of at least lizard_attn_fwd_workspace with
 *   dims.B = 1 (any L) but below that runs the sequences one after another.
 * Each sequence's results equal lizard_attn_fwd on that sequence alone: no state, window
 * or token crosses a sequence boundary.  With the larger workspace and the tensor-core
 * shapes (bf16, d = D = 128, four query heads per KV head, w = 64) every sequence is walked
 * in the same launches: its tokens are cut into segments of one length for the whole batch,
 * a (sequence x KV head, segment) CTA per segment, so a batch of many short sequences fills
 * the GPU as one long one does; other shapes run one sequence after another, each cut into
 * segments on its own.  Every sequence's slice must meet lizard_attn_fwd's 16-byte alignment
 * (for lse: Hq * 4 * cu_seqlens[i] a multiple of 16, true whenever Hq >= 4); errors are those
 * of lizard_attn_fwd, plus LIZARD_ERR_INVALID_ARG for inconsistent offsets. */
lizard_status lizard_attn_fwd_varlen(const lizard_dims* dims, const int64_t* cu_seqlens,
                                     const void* q, const void* k, const void* v, const void* g,
                                     const void* Wf, const float* sinks, void* y, float* lse,
                                     float* S_out, float* z_out, void* kcache_out,
                                     void* vcache_out, void* workspace, size_t ws_bytes,
                                     void* stream);

/* The forward for callers that cannot allocate device memory.  The Lizard pages have
 * no counterpart to this entry point; it exists for the integration.
 *
 * Some callers hold only pointers to their inputs and outputs: a plugin handed tensors
 * by a host framework that owns every device allocation, or a latency-critical loop that
 * must not call cudaMalloc/cudaFree because those can synchronise the whole device.  This
 * call takes no workspace.  It computes exactly what lizard_attn_fwd computes (the same
 * kernels in the same order, so the results are bit-identical), with the same arguments
 * minus the workspace and the same argument checks, and allocates nothing: its scratch (the
 * status word and the per-segment boundary states) is one 32 MiB array in device memory that
 * the library defines at file scope, so every GPU that loads the library holds those 32 MiB
 * until the process exits.
 *   - lizard_attn_fwd_noalloc_scratch(dims) gives the bytes of that array a call needs; a
 *     problem needing more than 32 MiB is rejected with LIZARD_ERR_WORKSPACE before anything
 *     is launched.
 *   - The first call on a device looks up the array's device address (with that device
 *     current) and caches it; make that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents: each call clears
 *     the status word on `stream` before its kernels, and every boundary record is written
 *     before it is read.  Calls whose work overlaps on the GPU (different streams, or
 *     different host threads) race on the array: order them on one stream.
 *   - A device-side error of a call (a bounded wait that gave up) is recorded in the array's
 *     status word; read it with lizard_read_noalloc_status after the call and before the
 *     next one (the next call clears it). */
lizard_status lizard_attn_fwd_noalloc(const lizard_dims* dims, const void* q, const void* k,
                                      const void* v, const void* g, const void* Wf,
                                      const float* sinks, void* y, float* lse, float* S_out,
                                      float* z_out, void* kcache_out, void* vcache_out,
                                      void* stream);

/* Bytes of lizard_attn_fwd_noalloc's 32 MiB array that a call with these sizes uses: 256
 * (status word) plus the boundary-state records of its launch, R * B * Hkv * (D*d + 2*D) * 4,
 * with R the number of records its segmentation writes (at least 1 on the tensor-core path,
 * 0 on the SIMT path when the sequence is one segment), plus, from the next 256-byte
 * boundary, the MASKED or LAGGED reading's scratch (one value per gate element); for the
 * MASKED reading the larger of its two walks' needs (see lizard_attn_fwd_kernel).  0 for
 * invalid sizes.  Pure host query; no counterpart on the Lizard pages. */
size_t lizard_attn_fwd_noalloc_scratch(const lizard_dims* dims);

/* Synchronise `stream`, read and clear the status word of lizard_attn_fwd_noalloc's array on
 * the current device.  Returns LIZARD_OK or the error a kernel of the last call recorded
 * (e.g. LIZARD_ERR_TIMEOUT).  No counterpart on the Lizard pages. */
lizard_status lizard_read_noalloc_status(void* stream);

/* Bytes of device workspace lizard_attn_bwd needs: segment records whose size depends on
 * B, Hkv, d and D only, plus one fp32 per gate element (B * L * Hkv * D * 4 bytes) holding
 * the per-position gate gradient before its reverse cumulative sum, plus two fp32 per query
 * row (e^{-lse} and dy . y, B * L * Hq * 8 bytes); the LAGGED reading adds one dtype value
 * per gate element (the moved gates), the MASKED reading two fp32 (the keys' log gate
 * products and their gate terms). */
size_t lizard_attn_bwd_workspace(const lizard_dims* dims);

/* Exact gradient of lizard_attn_fwd's y against an upstream gradient dy.  The
 * pages give no backward; this is the adjoint of the forward definition.
 *   y, lse        the forward's y and lse for the same inputs;
 *   dq, dk, dv, dg outputs in dtype; dWf [Hkv, d, D/2] and dsinks [Hq, M] fp32;
 *   every output is overwritten.  Reductions use a fixed order (deterministic). */
lizard_status lizard_attn_bwd(const lizard_dims* dims, const void* q, const void* k,
                              const void* v, const void* g, const void* Wf, const float* sinks,
                              const void* y, const float* lse, const void* dy, void* dq, void* dk,
                              void* dv, void* dg, float* dWf, float* dsinks, void* workspace,
                              size_t ws_bytes, void* stream);

/* Bytes of device workspace for lizard_attn_bwd_varlen on this packed batch (dims.B
 * sequences, dims.L tokens in all, host offsets cu_seqlens as for lizard_attn_fwd_varlen):
 * four lanes, each with the largest single-sequence backward workspace and room for one
 * sequence's dWf and dsinks and the lane's sums of them; 0 for inconsistent offsets.  A
 * quarter of it (one lane) is the least the call accepts. */
size_t lizard_attn_bwd_varlen_workspace(const lizard_dims* dims, const int64_t* cu_seqlens);

/* Backward of lizard_attn_fwd_varlen: packed q, k, v, g, y, dy, dq, dk, dv, dg [T, ...] and
 * lse [T, Hq] as in the forward; dWf [Hkv, d, D/2] and dsinks [Hq, M] fp32 are the sums over
 * the sequences.  Each sequence's dq, dk, dv, dg equal lizard_attn_bwd on that sequence
 * alone.  With the full lizard_attn_bwd_varlen_workspace the sequences run as independent
 * backwards on four streams of the library's own, forked from `stream` and joined back to it
 * before the call returns (longest sequences first, each to the lane with the fewest tokens
 * so far); each lane sums its sequences' dWf, dsinks in sequence order and the lanes are added
 * in lane order, so the result is deterministic for a given batch.  A workspace of one lane's
 * share runs the sequences one after another on `stream`, summed in sequence order.  Device
 * errors of every lane reach the status word at the head of `workspace`.  Errors as for
 * lizard_attn_bwd, plus LIZARD_ERR_INVALID_ARG for inconsistent offsets. */
lizard_status lizard_attn_bwd_varlen(const lizard_dims* dims, const int64_t* cu_seqlens,
                                     const void* q, const void* k, const void* v, const void* g,
                                     const void* Wf, const float* sinks, const void* y,
                                     const float* lse, const void* dy, void* dq, void* dk,
                                     void* dv, void* dg, float* dWf, float* dsinks,
                                     void* workspace, size_t ws_bytes, void* stream);

/* The projections in front of the mixer (sec. 2-A-1: the gate is a learned projection of
 * the layer input, Gamma_i = sigmoid(W_gamma x_i), next to the attention projections), as one
 * tensor-core GEMM:  [q | k | v | g] = x W^T.
 *   dims     the mixer's sizes (B, L, Hq, Hkv, d, D; the others are not used); dtype BF16;
 *   dmodel   width of the layer input, a multiple of 64;
 *   x        [B, L, dmodel] bf16;   W  [N, dmodel] bf16 with N = Hq d + 2 Hkv d + Hkv D, its rows
 *            q (Hq d), k (Hkv d), v (Hkv d), gate logits (Hkv D), each head's rows contiguous;
 *   q, k, v, g  outputs in the mixer's layouts ([B, L, Hq, d], [B, L, Hkv, d] x 2,
 *            [B, L, Hkv, D]), overwritten;
 *   workspace, ws_bytes  optional (NULL, 0): >= 256 bytes whose status word records a
 *            device-side error (read it with lizard_read_device_status).
 * Each of Hq d, Hkv d and Hkv D must be a multiple of 128, else LIZARD_ERR_UNSUPPORTED; fp32
 * dims also give LIZARD_ERR_UNSUPPORTED.  fp32 accumulation, bf16 results. */
lizard_status lizard_qkvg_proj(const lizard_dims* dims, int64_t dmodel, const void* x,
                               const void* W, void* q, void* k, void* v, void* g,
                               void* workspace, size_t ws_bytes, void* stream);

/* Backward of lizard_qkvg_proj from the mixer's gradients dq, dk, dv, dg (dY = [dq|dk|dv|dg]):
 *   dx [B, L, dmodel] bf16 = dY W,   dW [N, dmodel] fp32 = dY^T x   (both overwritten).
 * Sizes, layouts, workspace and errors as for lizard_qkvg_proj. */
lizard_status lizard_qkvg_proj_bwd(const lizard_dims* dims, int64_t dmodel, const void* x,
                                   const void* W, const void* dq, const void* dk,
                                   const void* dv, const void* dg, void* dx, float* dW,
                                   void* workspace, size_t ws_bytes, void* stream);

/* Bytes of device workspace lizard_decode_step needs: the status word, plus for the MASKED
 * and LAGGED readings B Hkv D values (the step's decay gates or key factors). */
size_t lizard_decode_workspace(const lizard_dims* dims);

/* Fill the gate ring a MASKED or LAGGED decode continues from: the gate logits of the last
 * min(L, w) tokens of a prefill go to slot t mod (w+1) of gcache [B, Hkv, w+1, D] (dtype),
 * other slots untouched, as lizard_attn_fwd writes kcache_out and vcache_out.  g [B, L, Hkv,
 * D] is the prefill's input.  The gates of the tokens in the window are what these two
 * readings decay with later: the lagged state takes the gate of token pos - w at step pos,
 * the masked reading the product of the gates of tokens pos - w + 1 .. pos.  After a packed
 * prefill (lizard_attn_fwd_varlen), call it once per sequence with dims.B = 1, dims.L = the
 * sequence's length, g at its first row and gcache at its ring.  Errors:
 * LIZARD_ERR_INVALID_ARG for bad dims or null/misaligned pointers. */
lizard_status lizard_gate_cache_fill(const lizard_dims* dims, const void* g, void* gcache,
                                     void* stream);

/* One constant-memory generation step for every sequence of the batch
 * (sec. 2-A-1: the state is updated incrementally, no growing KV cache;
 * sec. 4: generation at 32K keeps constant memory).
 *   dims.L is ignored; pos is the 0-based position of the new token (the same
 *   for the whole batch);
 *   q [B, Hq, d], k, v [B, Hkv, d], g [B, Hkv, D]: the new token;
 *   S, z: the state after token pos-1, updated IN PLACE to the state after pos
 *   (decay by Gamma_pos, then admit token pos-w read from the ring);
 *   kcache, vcache: ring caches holding tokens pos-w .. pos-1; the new k, v are
 *   written to slot pos mod (w+1) IN PLACE;
 *   gcache: the gate-logit ring of the same tokens (lizard_gate_cache_fill after a prefill),
 *   the new g written to slot pos mod (w+1) IN PLACE; required for the MASKED and LAGGED
 *   readings (LIZARD_ERR_INVALID_ARG when null), ignored and may be NULL for DELAYED.  The
 *   lagged state decays by the gate of token pos - w (none while pos < w), the masked
 *   reading admits token pos - w scaled by the product of the gates of pos - w + 1 .. pos;
 *   y [B, Hq, d]: the output of token pos. */
lizard_status lizard_decode_step(const lizard_dims* dims, int64_t pos, const void* q,
                                 const void* k, const void* v, const void* g, const void* Wf,
                                 const float* sinks, void* y, float* S, float* z, void* kcache,
                                 void* vcache, void* gcache, void* workspace, size_t ws_bytes,
                                 void* stream);

/* The same step with one position per sequence, for batches whose sequences have
 * different lengths (continuous batching).
 *   pos: DEVICE array [B] of int64, 8-byte aligned, read by the kernel when it runs (so a
 *   captured CUDA graph may be replayed after the positions are advanced on the device);
 *   sequence b is at position pos[b]: its state, ring slots and output follow
 *   lizard_decode_step at that position.  The library does not own or modify pos.
 *   A negative pos[b] records LIZARD_ERR_INVALID_ARG in the workspace status word (read it
 *   with lizard_read_device_status) and leaves sequence b's y, state and caches untouched;
 *   the other sequences are computed.  Host-side errors are those of lizard_decode_step,
 *   plus LIZARD_ERR_INVALID_ARG for a null or misaligned pos. */
lizard_status lizard_decode_step_positions(const lizard_dims* dims, const int64_t* pos,
                                           const void* q, const void* k, const void* v,
                                           const void* g, const void* Wf, const float* sinks,
                                           void* y, float* S, float* z, void* kcache,
                                           void* vcache, void* gcache, void* workspace,
                                           size_t ws_bytes, void* stream);

/* Synchronise `stream`, read the device status word of `workspace` and clear it.
 * Returns LIZARD_OK or the first error a kernel recorded (e.g. LIZARD_ERR_TIMEOUT). */
lizard_status lizard_read_device_status(void* workspace, void* stream);

/* Failure-path self-test: one CTA holds TMEM, waits on a barrier that never completes,
 * gives up after limit_cycles SM cycles (at most 4e9, about two seconds) exactly like the
 * tensor-core kernels' waits, records LIZARD_ERR_TIMEOUT in the workspace status word,
 * frees its TMEM and returns.  No fault, no hang: the context stays usable.  Read the
 * result with lizard_read_device_status.  workspace NULL targets the status word of
 * lizard_attn_fwd_noalloc's array instead (read it with lizard_read_noalloc_status). */
lizard_status lizard_selftest_wait_timeout(void* workspace, size_t ws_bytes,
                                           long long limit_cycles, void* stream);

/* Static description of a status code. */
const char* lizard_status_string(lizard_status s);

/* Measurement hook.  While set (non-NULL cudaEvent_t handles), every later
 * lizard_attn_fwd / lizard_attn_bwd call records `before` on its stream right
 * before its dominant kernel (the chunk walk) and `after` right after it, so a
 * caller can time that kernel alone with cudaEventElapsedTime.  NULL, NULL turns
 * it off.  Process-wide; not for concurrent use from several threads. */
lizard_status lizard_profile_events(void* before, void* after);

/* Library version string. */
const char* lizard_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LIZARD_H */
