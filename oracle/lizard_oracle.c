/*
 * Plain float64 CPU oracle of the Lizard hybrid token mixer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this code.  It shares no code, header,
 * table or helper with the CUDA library; the two meet only through the seeded
 * input generator.
 *
 * What it computes (Lizard summary, gist.science/ko/paper/2507.09025):
 *   - sec. 2-A-1 (gated linear attention): a data-dependent gate
 *     Gamma_i = sigmoid(.) decays a constant-size hidden state S_i that is
 *     updated token by token (constant-memory inference);
 *   - sec. 2-A-2 (anchor window attention): softmax attention over a sliding
 *     window restores local precision, and learnable meta-memory scalars t_m are
 *     added to the softmax denominator only (attention "sinks");
 *   - sec. 2-C (hardware-aware algorithm): the feature map is the non-negative
 *     Hedgehog map.
 * The closed form of the output, with one normaliser shared by both parts and
 * phi(x) = [softmax(x Wf), softmax(-x Wf)], is
 *   y_i = [phi(q_i) S_i + sum_win e^{s q_i.k_j} v_j]
 *       / [phi(q_i).z_i + sum_win e^{s q_i.k_j} + sum_m e^{t_m}].
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - a key leaves the window (i-w, i] at step i, enters the state undecayed,
 *     and is decayed by every later gate:
 *        S_i = Gamma_i (.) S_{i-1} + [i >= w] phi(k_{i-w}) v_{i-w}^T,
 *        z_i = Gamma_i (.) z_{i-1} + [i >= w] phi(k_{i-w});
 *     Gamma (.) S scales row f of S by Gamma_f;
 *   - two other readings of which gates decay a past key are kept as a switch
 *     (dims.reading; the pages fix none of the three), as weights of a key
 *     j <= i-w at query i and as recurrences of the state S_i that query i reads:
 *       0 delayed key (the default):  prod_{s=j+w+1..i} Gamma_s,
 *           S_i = Gamma_i (.) S_{i-1} + phi(k_{i-w}) v_{i-w}^T;
 *       1 masked full GLA:            prod_{s=j+1..i} Gamma_s,
 *           S_i = Gamma_i (.) S_{i-1} + c_{i-w} (.) phi(k_{i-w}) v_{i-w}^T,
 *           c_j = prod_{s=j+1..j+w} Gamma_s (the gates the key saw in the window);
 *       2 lagged state:               prod_{s=j+1..i-w} Gamma_s,
 *           S_i = Gamma_{i-w} (.) S_{i-1} + phi(k_{i-w}) v_{i-w}^T;
 *     S_i = 0 for i < w in all three, and z follows S with phi(k) in place of
 *     phi(k) v^T;
 *   - one Wf and one gate row per KV head; query head h uses KV head h / G;
 *   - the sinks are per query head and enter the denominator only.
 *
 * Everything is the naive recurrence with explicit products: no log space,
 * no chunking, no max shift in the window exponentials (fp64 covers the ranges
 * used).  Parallel over (batch, KV head) units, which are independent.
 *
 * Parity status: pinned (brute force on tiny inputs, hand-derived closed form,
 * library softmax attention, invariants, finite differences for the reverse
 * pass).
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    long B, L, Hq, Hkv, d, D, w, M;
    long reading; /* 0 delayed key, 1 masked full GLA, 2 lagged state */
    double scale;
} ora_dims;

/* Hedgehog map (sec. 2-C: non-negative feature map), phi = [softmax(u), softmax(-u)],
 * u = x Wf with Wf [d, D/2] row-major.  Also returns u when u_out is not NULL. */
static void ora_phi(const double *x, const double *Wf, long d, long D, double *phi,
                    double *u_out) {
    long H = D / 2;
    double *u = u_out ? u_out : (double *)malloc(sizeof(double) * H);
    for (long f = 0; f < H; ++f) u[f] = 0.0;
    for (long c = 0; c < d; ++c)
        for (long f = 0; f < H; ++f) u[f] += x[c] * Wf[c * H + f];
    double mx = -INFINITY, mn = INFINITY;
    for (long f = 0; f < H; ++f) {
        if (u[f] > mx) mx = u[f];
        if (u[f] < mn) mn = u[f];
    }
    double sp = 0.0, sn = 0.0;
    for (long f = 0; f < H; ++f) {
        phi[f] = exp(u[f] - mx);
        phi[H + f] = exp(-u[f] + mn);
        sp += phi[f];
        sn += phi[H + f];
    }
    for (long f = 0; f < H; ++f) {
        phi[f] /= sp;
        phi[H + f] /= sn;
    }
    if (!u_out) free(u);
}

static double ora_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* Row of the gate that decays the state at step i (-1: no decay at this step). */
static long decay_row(const ora_dims *p, long i) {
    if (p->reading == 2) return i >= p->w ? i - p->w : -1;
    return i;
}

/* c_f = prod_{s=i-w+1..i} sigmoid(g_{s,f}) for the key entering at step i under the
 * masked reading; gate row s of the unit is gates + s * stride. */
static void window_gate_product(const double *gates, long stride, long i, long w, long D,
                                double *c) {
    for (long f = 0; f < D; ++f) c[f] = 1.0;
    for (long s = i - w + 1; s <= i; ++s)
        for (long f = 0; f < D; ++f) c[f] *= ora_sigmoid(gates[s * stride + f]);
}

static double dot(const double *a, const double *b, long n) {
    double s = 0.0;
    for (long i = 0; i < n; ++i) s += a[i] * b[i];
    return s;
}

/* Forward of the whole sequence by the token recurrence (sec. 2-A-1 and 2-A-2).
 * q [B,L,Hq,d]; k, v [B,L,Hkv,d]; g [B,L,Hkv,D]; Wf [Hkv,d,D/2]; sinks [Hq,M].
 * y [B,L,Hq,d].  Optional (NULL to skip):
 *   S_out [B,Hkv,D,d], z_out [B,Hkv,D]   final state after token L-1,
 *   num_gla [B,L,Hq,d], den_gla [B,L,Hq] the state's readout phi(q).S, phi(q).z,
 *   num_win [B,L,Hq,d], den_win [B,L,Hq] the window sums (no shift),
 *   den [B,L,Hq]                          the full shared denominator. */
int ora_fwd(const ora_dims *p, const double *q, const double *k, const double *v,
            const double *g, const double *Wf, const double *sinks, double *y, double *S_out,
            double *z_out, double *num_gla, double *den_gla, double *num_win, double *den_win,
            double *den_out) {
    const long B = p->B, L = p->L, Hq = p->Hq, Hkv = p->Hkv, d = p->d, D = p->D, w = p->w,
               M = p->M;
    if (Hkv <= 0 || Hq % Hkv != 0 || D % 2 != 0 || w < 1 || p->reading < 0 ||
        p->reading > 2)
        return 1;
    const long G = Hq / Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (long unit = 0; unit < B * Hkv; ++unit) {
        const long b = unit / Hkv, kv = unit % Hkv;
        const double *Wk = Wf + kv * d * (D / 2);
        double *S = (double *)calloc((size_t)(D * d), sizeof(double));
        double *z = (double *)calloc((size_t)D, sizeof(double));
        double *phk = (double *)malloc(sizeof(double) * D);
        double *phq = (double *)malloc(sizeof(double) * D);
        double *cf = (double *)malloc(sizeof(double) * D);
        double *num = (double *)malloc(sizeof(double) * d);
        const double *gu = g + (b * L * Hkv + kv) * D; /* gate row s: gu + s * Hkv * D */
        for (long i = 0; i < L; ++i) {
            /* decay by the reading's gate (Gamma_i, or Gamma_{i-w} for the lagged state),
             * then admit the key leaving the window */
            const long gr = decay_row(p, i);
            for (long f = 0; gr >= 0 && f < D; ++f) {
                double gam = ora_sigmoid(gu[gr * Hkv * D + f]);
                for (long c = 0; c < d; ++c) S[f * d + c] *= gam;
                z[f] *= gam;
            }
            if (i >= w) {
                const double *kx = k + ((b * L + (i - w)) * Hkv + kv) * d;
                const double *vx = v + ((b * L + (i - w)) * Hkv + kv) * d;
                ora_phi(kx, Wk, d, D, phk, NULL);
                if (p->reading == 1) {
                    window_gate_product(gu, Hkv * D, i, w, D, cf);
                    for (long f = 0; f < D; ++f) phk[f] *= cf[f];
                }
                for (long f = 0; f < D; ++f) {
                    for (long c = 0; c < d; ++c) S[f * d + c] += phk[f] * vx[c];
                    z[f] += phk[f];
                }
            }
            for (long hh = 0; hh < G; ++hh) {
                const long h = kv * G + hh;
                const double *qi = q + ((b * L + i) * Hq + h) * d;
                ora_phi(qi, Wk, d, D, phq, NULL);
                for (long c = 0; c < d; ++c) num[c] = 0.0;
                for (long f = 0; f < D; ++f)
                    for (long c = 0; c < d; ++c) num[c] += phq[f] * S[f * d + c];
                double dg_ = dot(phq, z, D);
                const long row = (b * L + i) * Hq + h;
                if (num_gla)
                    for (long c = 0; c < d; ++c) num_gla[row * d + c] = num[c];
                if (den_gla) den_gla[row] = dg_;
                double dw = 0.0;
                double *nw = num_win ? num_win + row * d : NULL;
                if (nw)
                    for (long c = 0; c < d; ++c) nw[c] = 0.0;
                long j0 = i - w + 1 < 0 ? 0 : i - w + 1;
                for (long j = j0; j <= i; ++j) {
                    const double *kj = k + ((b * L + j) * Hkv + kv) * d;
                    const double *vj = v + ((b * L + j) * Hkv + kv) * d;
                    double e = exp(p->scale * dot(qi, kj, d));
                    for (long c = 0; c < d; ++c) num[c] += e * vj[c];
                    if (nw)
                        for (long c = 0; c < d; ++c) nw[c] += e * vj[c];
                    dw += e;
                }
                if (den_win) den_win[row] = dw;
                double sk = 0.0;
                for (long m = 0; m < M; ++m) sk += exp(sinks[h * M + m]);
                double den = dg_ + dw + sk;
                if (den_out) den_out[row] = den;
                for (long c = 0; c < d; ++c) y[row * d + c] = num[c] / den;
            }
        }
        if (S_out) memcpy(S_out + unit * D * d, S, sizeof(double) * D * d);
        if (z_out) memcpy(z_out + unit * D, z, sizeof(double) * D);
        free(S);
        free(z);
        free(phk);
        free(phq);
        free(cf);
        free(num);
    }
    return 0;
}

/* One decode step at position pos for every sequence of the batch (sec. 2-A-1,
 * constant-memory inference).  q [B,Hq,d]; k, v [B,Hkv,d]; g [B,Hkv,D] hold the
 * new token.  S [B,Hkv,D,d] and z [B,Hkv,D] hold the state after token pos-1 and
 * are updated in place.  kc, vc [B,Hkv,w+1,d] are ring caches: token t lives in
 * slot t mod (w+1); the new token is written to its slot.  y [B,Hq,d].
 * gc [B,Hkv,w+1,D] is the same ring for the gate logits, which the masked and lagged
 * readings need (they decay or weigh with gates of tokens already in the window); it
 * may be NULL under the delayed-key reading. */
int ora_decode_step(const ora_dims *p, long pos, const double *q, const double *k,
                    const double *v, const double *g, const double *Wf, const double *sinks,
                    double *y, double *S, double *z, double *kc, double *vc, double *gc) {
    const long B = p->B, Hq = p->Hq, Hkv = p->Hkv, d = p->d, D = p->D, w = p->w, M = p->M;
    if (Hkv <= 0 || Hq % Hkv != 0 || D % 2 != 0 || w < 1 || pos < 0) return 1;
    if (p->reading < 0 || p->reading > 2 || (p->reading != 0 && gc == NULL)) return 1;
    const long G = Hq / Hkv, R = w + 1;
#pragma omp parallel for schedule(dynamic, 1)
    for (long unit = 0; unit < B * Hkv; ++unit) {
        const long b = unit / Hkv, kv = unit % Hkv;
        const double *Wk = Wf + kv * d * (D / 2);
        double *Su = S + unit * D * d, *zu = z + unit * D;
        double *kcu = kc + unit * R * d, *vcu = vc + unit * R * d;
        double *gcu = gc ? gc + unit * R * D : NULL;
        const double *gi = g + unit * D;
        double *phk = (double *)malloc(sizeof(double) * D);
        double *phq = (double *)malloc(sizeof(double) * D);
        double *num = (double *)malloc(sizeof(double) * d);
        /* the gate of this step: Gamma_pos, or Gamma_{pos-w} from the ring (lagged state) */
        const double *gd = gi;
        if (p->reading == 2) gd = pos >= w ? gcu + ((pos - w) % R) * D : NULL;
        for (long f = 0; gd != NULL && f < D; ++f) {
            double gam = ora_sigmoid(gd[f]);
            for (long c = 0; c < d; ++c) Su[f * d + c] *= gam;
            zu[f] *= gam;
        }
        if (pos >= w) {
            const long slot = (pos - w) % R;
            ora_phi(kcu + slot * d, Wk, d, D, phk, NULL);
            if (p->reading == 1) /* c = prod of the gates of tokens pos-w+1 .. pos */
                for (long s = pos - w + 1; s <= pos; ++s) {
                    const double *gs = s == pos ? gi : gcu + (s % R) * D;
                    for (long f = 0; f < D; ++f) phk[f] *= ora_sigmoid(gs[f]);
                }
            for (long f = 0; f < D; ++f) {
                for (long c = 0; c < d; ++c) Su[f * d + c] += phk[f] * vcu[slot * d + c];
                zu[f] += phk[f];
            }
        }
        /* the new token joins the ring before the window is read */
        memcpy(kcu + (pos % R) * d, k + unit * d, sizeof(double) * d);
        memcpy(vcu + (pos % R) * d, v + unit * d, sizeof(double) * d);
        if (gcu) memcpy(gcu + (pos % R) * D, gi, sizeof(double) * D);
        for (long hh = 0; hh < G; ++hh) {
            const long h = kv * G + hh;
            const double *qi = q + (b * Hq + h) * d;
            ora_phi(qi, Wk, d, D, phq, NULL);
            for (long c = 0; c < d; ++c) num[c] = 0.0;
            for (long f = 0; f < D; ++f)
                for (long c = 0; c < d; ++c) num[c] += phq[f] * Su[f * d + c];
            double den = dot(phq, zu, D);
            long j0 = pos - w + 1 < 0 ? 0 : pos - w + 1;
            for (long j = j0; j <= pos; ++j) {
                const double *kj = kcu + (j % R) * d, *vj = vcu + (j % R) * d;
                double e = exp(p->scale * dot(qi, kj, d));
                for (long c = 0; c < d; ++c) num[c] += e * vj[c];
                den += e;
            }
            for (long m = 0; m < M; ++m) den += exp(sinks[h * M + m]);
            for (long c = 0; c < d; ++c) y[(b * Hq + h) * d + c] = num[c] / den;
        }
        free(phk);
        free(phq);
        free(num);
    }
    return 0;
}

/* Reverse of the Hedgehog map: given x, dphi, accumulate dx (+=) and dWf (+=). */
static void ora_phi_bwd(const double *x, const double *Wk, long d, long D, const double *dphi,
                        double *dx, double *dWk) {
    long H = D / 2;
    double *phi = (double *)malloc(sizeof(double) * D);
    double *du = (double *)malloc(sizeof(double) * H);
    ora_phi(x, Wk, d, D, phi, NULL);
    double sp = 0.0, sn = 0.0;
    for (long f = 0; f < H; ++f) {
        sp += phi[f] * dphi[f];
        sn += phi[H + f] * dphi[H + f];
    }
    /* d softmax(u) = p (dp - p.dp); softmax(-u) contributes with a minus sign */
    for (long f = 0; f < H; ++f)
        du[f] = phi[f] * (dphi[f] - sp) - phi[H + f] * (dphi[H + f] - sn);
    for (long c = 0; c < d; ++c)
        for (long f = 0; f < H; ++f) {
            dx[c] += Wk[c * H + f] * du[f];
            dWk[c * H + f] += x[c] * du[f];
        }
    free(phi);
    free(du);
}

/* Transition of step i on one unit's augmented state [S | z] (D x (d+1)), under the
 * dims' reading: cur = gamma (.) prev + [i >= w] a (.) phi(k_{i-w}) [v_{i-w} | 1], with gamma
 * the gate of decay_row(i) (1 when there is none) and a = c_{i-w} (masked reading) or 1.
 * gu: gate row 0 of the unit (row s at gu + s * gstride); kx, vx: key and value i-w.
 * cur may be prev.  phk, cf: scratch [D]. */
static void ora_transition(const ora_dims *p, const double *gu, long gstride, const double *kx,
                           const double *vx, const double *Wk, long i, const double *prev,
                           double *cur, double *phk, double *cf) {
    const long d = p->d, D = p->D, w = p->w, E = d + 1;
    const long gr = decay_row(p, i);
    for (long f = 0; f < D; ++f) {
        double gam = gr >= 0 ? ora_sigmoid(gu[gr * gstride + f]) : 1.0;
        for (long c = 0; c < E; ++c) cur[f * E + c] = gam * prev[f * E + c];
    }
    if (i < w) return;
    ora_phi(kx, Wk, d, D, phk, NULL);
    if (p->reading == 1) {
        window_gate_product(gu, gstride, i, w, D, cf);
        for (long f = 0; f < D; ++f) phk[f] *= cf[f];
    }
    for (long f = 0; f < D; ++f) {
        for (long c = 0; c < d; ++c) cur[f * E + c] += phk[f] * vx[c];
        cur[f * E + d] += phk[f];
    }
}

/* Exact gradient of ora_fwd (the pages give no backward; this is the adjoint of
 * the same recurrence).  The augmented state [S | z] (D x (d+1)) is checkpointed
 * every 64 tokens and recomputed one block at a time in the reverse sweep.
 * Outputs dq [B,L,Hq,d], dk, dv [B,L,Hkv,d], dg [B,L,Hkv,D], dWf [Hkv,d,D/2],
 * dsinks [Hq,M]; every output is overwritten. */
int ora_bwd(const ora_dims *p, const double *q, const double *k, const double *v,
            const double *g, const double *Wf, const double *sinks, const double *dy,
            double *dq, double *dk, double *dv, double *dg, double *dWf, double *dsinks) {
    const long B = p->B, L = p->L, Hq = p->Hq, Hkv = p->Hkv, d = p->d, D = p->D, w = p->w,
               M = p->M;
    if (Hkv <= 0 || Hq % Hkv != 0 || D % 2 != 0 || w < 1 || p->reading < 0 ||
        p->reading > 2)
        return 1;
    const long G = Hq / Hkv, E = d + 1, CK = 64;
    const long nblk = (L + CK - 1) / CK;
    const long wsz = d * (D / 2);
    double *dWpart = (double *)calloc((size_t)(B * Hkv * wsz), sizeof(double));
    double *dtpart = (double *)calloc((size_t)(B * Hkv * G * M), sizeof(double));
    memset(dq, 0, sizeof(double) * B * L * Hq * d);
    memset(dk, 0, sizeof(double) * B * L * Hkv * d);
    memset(dv, 0, sizeof(double) * B * L * Hkv * d);
    memset(dg, 0, sizeof(double) * B * L * Hkv * D);
#pragma omp parallel for schedule(dynamic, 1)
    for (long unit = 0; unit < B * Hkv; ++unit) {
        const long b = unit / Hkv, kv = unit % Hkv;
        const double *Wk = Wf + kv * wsz;
        double *dWk = dWpart + unit * wsz;
        double *dtk = dtpart + unit * G * M;
#define KIDX(t) (((b * L + (t)) * Hkv + kv) * d)
#define GIDX(t) (((b * L + (t)) * Hkv + kv) * D)
        /* checkpoints: ck[blk] = augmented state after token blk*CK - 1 */
        double *ck = (double *)calloc((size_t)(nblk * D * E), sizeof(double));
        double *St = (double *)calloc((size_t)(D * E), sizeof(double));
        double *phk = (double *)malloc(sizeof(double) * D);
        double *cf = (double *)malloc(sizeof(double) * D);
        const double *gu = g + GIDX(0);
        const long gs = Hkv * D;
        for (long i = 0; i < L; ++i) {
            if (i % CK == 0) memcpy(ck + (i / CK) * D * E, St, sizeof(double) * D * E);
            const long j = i >= w ? i - w : 0;
            ora_transition(p, gu, gs, k + KIDX(j), v + KIDX(j), Wk, i, St, St, phk, cf);
        }
        /* reverse sweep; Gb = gradient w.r.t. the augmented state after token i */
        double *Gb = (double *)calloc((size_t)(D * E), sizeof(double));
        double *blk = (double *)malloc(sizeof(double) * (size_t)((CK + 1) * D * E));
        double *phq = (double *)malloc(sizeof(double) * D);
        double *dph = (double *)malloc(sizeof(double) * D);
        double *num = (double *)malloc(sizeof(double) * d);
        double *dnum = (double *)malloc(sizeof(double) * d);
        double *pw = (double *)malloc(sizeof(double) * (size_t)w);
        for (long bi = nblk - 1; bi >= 0; --bi) {
            const long i0 = bi * CK, i1 = (i0 + CK < L) ? i0 + CK : L;
            /* blk[0] = state after i0-1; blk[t+1] = state after i0+t */
            memcpy(blk, ck + bi * D * E, sizeof(double) * D * E);
            for (long i = i0; i < i1; ++i) {
                double *prev = blk + (i - i0) * D * E, *cur = prev + D * E;
                const long j = i >= w ? i - w : 0;
                ora_transition(p, gu, gs, k + KIDX(j), v + KIDX(j), Wk, i, prev, cur, phk, cf);
            }
            for (long i = i1 - 1; i >= i0; --i) {
                const double *prev = blk + (i - i0) * D * E, *cur = prev + D * E;
                /* outputs of token i */
                for (long hh = 0; hh < G; ++hh) {
                    const long h = kv * G + hh;
                    const long row = (b * L + i) * Hq + h;
                    const double *qi = q + row * d;
                    const double *dyi = dy + row * d;
                    ora_phi(qi, Wk, d, D, phq, NULL);
                    for (long c = 0; c < d; ++c) num[c] = 0.0;
                    double den = 0.0;
                    for (long f = 0; f < D; ++f) {
                        for (long c = 0; c < d; ++c) num[c] += phq[f] * cur[f * E + c];
                        den += phq[f] * cur[f * E + d];
                    }
                    long j0 = i - w + 1 < 0 ? 0 : i - w + 1;
                    for (long j = j0; j <= i; ++j) {
                        double e = exp(p->scale * dot(qi, k + KIDX(j), d));
                        pw[j - j0] = e;
                        const double *vj = v + KIDX(j);
                        for (long c = 0; c < d; ++c) num[c] += e * vj[c];
                        den += e;
                    }
                    for (long m = 0; m < M; ++m) den += exp(sinks[h * M + m]);
                    /* y = num/den: dnum = dy/den, dden = -(dy.y)/den */
                    double delta = 0.0;
                    for (long c = 0; c < d; ++c) delta += dyi[c] * num[c] / den;
                    for (long c = 0; c < d; ++c) dnum[c] = dyi[c] / den;
                    double dden = -delta / den;
                    for (long m = 0; m < M; ++m) dtk[hh * M + m] += exp(sinks[h * M + m]) * dden;
                    /* window: s = scale q.k, e = exp(s) */
                    double *dqi = dq + row * d;
                    for (long j = j0; j <= i; ++j) {
                        const double *vj = v + KIDX(j), *kj = k + KIDX(j);
                        double e = pw[j - j0];
                        double ds = e * (dot(dnum, vj, d) + dden);
                        double *dvj = dv + KIDX(j), *dkj = dk + KIDX(j);
                        for (long c = 0; c < d; ++c) {
                            dvj[c] += e * dnum[c];
                            dqi[c] += p->scale * ds * kj[c];
                            dkj[c] += p->scale * ds * qi[c];
                        }
                    }
                    /* state readout phi(q).[S | z] */
                    for (long f = 0; f < D; ++f) {
                        double s = 0.0;
                        for (long c = 0; c < d; ++c) {
                            s += cur[f * E + c] * dnum[c];
                            Gb[f * E + c] += phq[f] * dnum[c];
                        }
                        s += cur[f * E + d] * dden;
                        Gb[f * E + d] += phq[f] * dden;
                        dph[f] = s;
                    }
                    ora_phi_bwd(qi, Wk, d, D, dph, dqi, dWk);
                }
                /* state update of token i: cur = gamma (.) prev + [i>=w] a (.) phi(k_{i-w}) [v | 1]
                 * (ora_transition); gamma's gate row gets dgamma gamma (1 - gamma) */
                const long gr = decay_row(p, i);
                if (gr >= 0) {
                    const double *gg = g + GIDX(gr);
                    double *dgr = dg + GIDX(gr);
                    for (long f = 0; f < D; ++f) {
                        double gam = ora_sigmoid(gg[f]);
                        double s = 0.0;
                        for (long c = 0; c < E; ++c) s += Gb[f * E + c] * prev[f * E + c];
                        dgr[f] += s * gam * (1.0 - gam);
                    }
                }
                if (i >= w) {
                    const double *kx = k + KIDX(i - w), *vx = v + KIDX(i - w);
                    double *dvx = dv + KIDX(i - w), *dkx = dk + KIDX(i - w);
                    ora_phi(kx, Wk, d, D, phk, NULL);
                    for (long f = 0; f < D; ++f) cf[f] = 1.0;
                    if (p->reading == 1) window_gate_product(gu, gs, i, w, D, cf);
                    for (long f = 0; f < D; ++f) {
                        /* s = d/d(a phi_f); the value sees a phi_f */
                        double s = Gb[f * E + d];
                        for (long c = 0; c < d; ++c) {
                            s += Gb[f * E + c] * vx[c];
                            dvx[c] += Gb[f * E + c] * cf[f] * phk[f];
                        }
                        dph[f] = cf[f] * s;
                        /* masked reading: a_f = prod_{u=i-w+1..i} Gamma_u, so each of those
                         * gates gets (a phi_f s) (1 - Gamma_u) */
                        if (p->reading == 1) {
                            const double da = cf[f] * phk[f] * s;
                            for (long u = i - w + 1; u <= i; ++u)
                                dg[GIDX(u) + f] += da * (1.0 - ora_sigmoid(g[GIDX(u) + f]));
                        }
                    }
                    ora_phi_bwd(kx, Wk, d, D, dph, dkx, dWk);
                }
                if (gr >= 0) {
                    const double *gg = g + GIDX(gr);
                    for (long f = 0; f < D; ++f) {
                        double gam = ora_sigmoid(gg[f]);
                        for (long c = 0; c < E; ++c) Gb[f * E + c] *= gam;
                    }
                }
            }
        }
#undef KIDX
#undef GIDX
        free(ck);
        free(St);
        free(phk);
        free(cf);
        free(Gb);
        free(blk);
        free(phq);
        free(dph);
        free(num);
        free(dnum);
        free(pw);
    }
    /* deterministic reductions over the batch */
    memset(dWf, 0, sizeof(double) * Hkv * wsz);
    memset(dsinks, 0, sizeof(double) * Hq * M);
    for (long b = 0; b < B; ++b)
        for (long kv = 0; kv < Hkv; ++kv) {
            const long unit = b * Hkv + kv;
            for (long e = 0; e < wsz; ++e) dWf[kv * wsz + e] += dWpart[unit * wsz + e];
            for (long hh = 0; hh < G; ++hh)
                for (long m = 0; m < M; ++m)
                    dsinks[(kv * G + hh) * M + m] += dtpart[(unit * G + hh) * M + m];
        }
    free(dWpart);
    free(dtpart);
    return 0;
}
