/*
 * moe_oracle.c -- plain, slow CPU oracle for one MoE routing layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg load this file's library.  The GPU library never links,
 * includes or calls it, and it shares no code, header, table or constant with
 * the GPU path.  Build with -ffp-contract=off so that every fp32 product and
 * sum is rounded on its own, exactly as written.
 *
 * Sources (cited by page title and section):
 *   [MACS]  "MACS: Modality-Aware Capacity Scaling for Efficient Multimodal MoE
 *           Inference", sections 3.1-3.3, Eqs. (1)-(7).
 *   [SERE]  Xiaohongshu engineering article on multi-image QA inference
 *           ("dynamic visual token compression + SERE expert rerouting"),
 *           section 4.1 (algorithm) and 4.2 (engineering, critical-expert
 *           protection).
 *
 * Threads: the router, the FFN + combine and the similarity calibration loop
 * over independent tokens or experts with OpenMP (orc_set_threads).  Each
 * output element is computed by one thread in the order written, so results
 * are identical for every thread count.
 *
 * Precision: everything the layer computes in floating point is done in
 * double, except the steps whose result decides an integer (the ranking, the
 * gates that order capacity admission, the similarity threshold, the merged
 * gate) -- those are done in fp32 with the operation order stated beside
 * them, because the GPU path takes the same decisions in fp32.
 *
 * Parity status per function (pins live in tests/test_oracle_*.py):
 *   orc_exp_spec       pinned: within 2 ulp of exp() on sampled inputs; constants
 *                      re-derived from exact rationals.
 *   orc_router         pinned: numpy float64 matmul.
 *   orc_route          pinned: ranking vs numpy lexsort; gates vs exact softmax.
 *   orc_sere           pinned: closed forms (rho>1, K'=k), invariants, a
 *                      declarative property check, hand-worked golden cases.
 *   orc_capacity       pinned: w==1 reduces to Eq. (3) count capacity, huge
 *                      gamma reduces to plain dispatch, declarative brute force,
 *                      hand-worked golden case.  Per-expert capacity (a
 *                      reading of the truncated [MACS] 3.3): m = 0 or
 *                      R_v = 1/2 reduce to the static case, unit weights give
 *                      floor(gamma T k / N (1 + m (R_v - 1/2))) tokens (exact
 *                      rationals), declarative brute force per expert.
 *   orc_permute        pinned: numpy lexsort on (expert, token).
 *   orc_ffn_combine    pinned: dense numpy float64 evaluation of Eq. (1).
 *   orc_similarity     pinned: a duplicated expert -> 1, a negated down
 *                      projection -> -1, a positively scaled one -> 1,
 *                      experts writing disjoint coordinates -> 0, symmetry,
 *                      unit diagonal, |sim| <= 1; closed forms for the
 *                      SwiGLU orientation (-1), the stacked-token cosine
 *                      (1/sqrt 2) and the sign of silu(c) + silu(-c).
 *   orc_token_weights  pinned: entropy against scipy's entropy of softmax,
 *                      closed forms (uniform z -> ln D, one raised entry,
 *                      shift invariance), two-token z-score -> sigmoid(+-delta),
 *                      text weight 1, delta = 0 -> 1/2, R_v bounds.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_EINVAL -1
#define ORC_ENONFINITE -2
#define ORC_ENOMEM -3

#define ORC_DT_F32 0
#define ORC_DT_BF16 1

#define ORC_SLOT_KEPT 0
#define ORC_SLOT_REROUTED 1
#define ORC_SLOT_DROPPED 2

/* ------------------------------------------------------------------ */
/* Deterministic fp32 exponential for non-positive arguments.           */
/*                                                                      */
/* The gates must be reproducible bit for bit because capacity          */
/* admission orders tokens by gate.  The method: Cody & Waite range     */
/* reduction d = n ln2 + r with ln2 split into a head with 15           */
/* significant bits (n ln2_hi exact for |n| < 512) and a tail, then     */
/* the degree-7 Taylor polynomial of e^r in Horner form with fused      */
/* multiply-adds, then an exact scaling by 2^n.  Results that would be  */
/* subnormal (n < -125) are flushed to zero.                            */
/* ------------------------------------------------------------------ */
static const float ORC_LOG2E = 0x1.715476p+0f;      /* log2(e) rounded to fp32 */
static const float ORC_LN2_HI = 0x1.62e4p-1f;       /* floor(ln2 * 2^15) / 2^15 = 22713/32768 */
static const float ORC_LN2_LO = 0x1.7f7d1cp-20f;    /* ln2 - LN2_HI rounded to fp32 */
static const float ORC_INV_FACT[8] = {              /* 1/i! rounded to fp32 */
    0x1p+0f, 0x1p+0f, 0x1p-1f, 0x1.555556p-3f,
    0x1.555556p-5f, 0x1.111112p-7f, 0x1.6c16c2p-10f, 0x1.a01a02p-13f};

float orc_exp_spec(float d) {
    float n = rintf(d * ORC_LOG2E);
    if (n < -125.0f) return 0.0f;
    float r = fmaf(-n, ORC_LN2_HI, d);
    r = fmaf(-n, ORC_LN2_LO, r);
    float p = ORC_INV_FACT[7];
    for (int i = 6; i >= 0; --i) p = fmaf(p, r, ORC_INV_FACT[i]);
    /* 2^n as an fp32 bit pattern; exact product because the result is normal */
    int ni = (int)n;
    uint32_t bits = (uint32_t)(ni + 127) << 23;
    float scale;
    memcpy(&scale, &bits, sizeof scale);
    return p * scale;
}

void orc_exp_spec_array(const float* d, float* out, long n) {
    for (long i = 0; i < n; ++i) out[i] = orc_exp_spec(d[i]);
}

/* Exposes the constants so that a test can re-derive them independently. */
void orc_exp_constants(float out[11]) {
    out[0] = ORC_LOG2E;
    out[1] = ORC_LN2_HI;
    out[2] = ORC_LN2_LO;
    for (int i = 0; i < 8; ++i) out[3 + i] = ORC_INV_FACT[i];
}

static double ld_val(const void* p, int dtype, size_t i) {
    if (dtype == ORC_DT_F32) return (double)((const float*)p)[i];
    uint32_t b = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    memcpy(&f, &b, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------ */
/* Router G(x): logits[t][j] = sum_h x[t][h] * w_r[j][h]                */
/* [MACS] 3.1, the router network that scores every expert for a token. */
/* Accumulated in double, stored as fp32.                               */
/* ------------------------------------------------------------------ */
int orc_router(const void* x, int x_dtype, const float* w_r, int T, int H, int N, float* logits) {
    if (!x || !w_r || !logits || T < 0 || H <= 0 || N <= 0) return ORC_EINVAL;
    /* tokens are independent: each thread owns whole rows of logits, and the
       sum over h runs in the same order whatever the thread count */
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < N; ++j) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += ld_val(x, x_dtype, (size_t)t * H + h) * (double)w_r[(size_t)j * H + h];
            logits[(size_t)t * N + j] = (float)acc;
        }
    return ORC_OK;
}

/* Host threads used by the loops over independent tokens or experts (the
   router, the FFN + combine, the similarity calibration's expert outputs).
   Results do not depend on it: every output element is computed by one
   thread in the order written.  n <= 0 selects every host core. */
void orc_set_threads(int n) {
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : omp_get_num_procs());
#else
    (void)n;
#endif
}

int orc_get_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ */
/* Softmax gate and top-R ranking.  [MACS] 3.1 Eq. (1): the layer keeps  */
/* the top-k experts of G(x) and weights each by its gate G(x)_j.        */
/*                                                                      */
/* Gate (fp32, fixed order):                                            */
/*   m = max_j l_j; e_j = exp_spec(l_j - m);                            */
/*   Z: 32 partial sums, partial[l] = e_l + e_{l+32} + ... in order,    */
/*      then five butterfly rounds partial[l] += partial[l ^ off] for    */
/*      off = 16, 8, 4, 2, 1 (all lanes updated from the previous        */
/*      round's values); Z = partial[0];                                */
/*   g_j = e_j / Z.                                                     */
/* Ranking: by logit descending, ties to the lower expert id.           */
/* renorm_k > 0 divides the first renorm_k gates by their sequential    */
/* fp32 sum (an option; Eq. (1) uses the raw gate).                     */
/* ------------------------------------------------------------------ */
int orc_route(const float* logits, int T, int N, int R, int renorm_k, int32_t* ids, float* gates) {
    if (!logits || !ids || !gates || T < 0 || N <= 0 || R <= 0 || R > N || renorm_k < 0 || renorm_k > R)
        return ORC_EINVAL;
    float* e = (float*)malloc(sizeof(float) * (size_t)N);
    unsigned char* taken = (unsigned char*)malloc((size_t)N);
    if (!e || !taken) { free(e); free(taken); return ORC_ENOMEM; }
    int rc = ORC_OK;
    for (int t = 0; t < T; ++t) {
        const float* l = logits + (size_t)t * N;
        float m = l[0];
        for (int j = 0; j < N; ++j) {
            if (!isfinite(l[j])) rc = ORC_ENONFINITE;
            if (l[j] > m) m = l[j];
        }
        if (rc != ORC_OK) break;
        for (int j = 0; j < N; ++j) e[j] = orc_exp_spec(l[j] - m);
        float partial[32];
        for (int ln = 0; ln < 32; ++ln) {
            float s = 0.0f;
            for (int j = ln; j < N; j += 32) s = s + e[j];
            partial[ln] = s;
        }
        for (int off = 16; off >= 1; off >>= 1) {
            float nxt[32];
            for (int ln = 0; ln < 32; ++ln) nxt[ln] = partial[ln] + partial[ln ^ off];
            memcpy(partial, nxt, sizeof partial);
        }
        float Z = partial[0];
        memset(taken, 0, (size_t)N);
        for (int r = 0; r < R; ++r) {
            int best = -1;
            for (int j = 0; j < N; ++j) {
                if (taken[j]) continue;
                if (best < 0 || l[j] > l[best]) best = j;   /* strict: lower id wins ties */
            }
            taken[best] = 1;
            ids[(size_t)t * R + r] = best;
            gates[(size_t)t * R + r] = e[best] / Z;
        }
        if (renorm_k > 0) {
            float s = 0.0f;
            for (int r = 0; r < renorm_k; ++r) s = s + gates[(size_t)t * R + r];
            for (int r = 0; r < renorm_k; ++r) gates[(size_t)t * R + r] = gates[(size_t)t * R + r] / s;
        }
    }
    free(e);
    free(taken);
    return rc;
}

/* ------------------------------------------------------------------ */
/* SERE batch reroute.  [SERE] 4.1 and 4.2.                            */
/*                                                                      */
/* P = union over the batch of every token's top-K' (primary) experts.  */
/* For each token, secondary slots r = K'..k-1 in rank order, source    */
/* s = ids[t][r]:                                                       */
/*   - s protected ([SERE] 4.2: protection blocks only the source) or  */
/*     s already in P: keep;                                            */
/*   - else p* = argmax_{p in P} sim[s][p] (ties to the lower id); if    */
/*     sim[s][p*] > rho (strictly exceeds), the slot moves to p*; if the */
/*     token already holds p* in slot q, the gate is added to slot q     */
/*     (fp32 add) and slot r becomes empty (-1, 0);                     */
/*   - else keep (too dissimilar).                                      */
/* The candidate set is P alone, so a protected or kept secondary never */
/* attracts others.                                                     */
/* stats: [0] union before (top-k), [1] |P|, [2] union after,           */
/*        [3] moved, [4] merged, [5] kept: protected, [6] kept: sim<=rho */
/* ------------------------------------------------------------------ */
int orc_sere(int32_t* ids, float* gates, int ld, int T, int N, int k, int kp, float rho,
             const float* sim, const uint8_t* protect, uint32_t* bitmap, int32_t* stats) {
    if (!ids || !gates || !sim || T < 0 || N <= 0 || k <= 0 || ld < k || kp < 1 || kp > k) return ORC_EINVAL;
    unsigned char* inP = (unsigned char*)calloc((size_t)N, 1);
    unsigned char* seen = (unsigned char*)calloc((size_t)N, 1);
    if (!inP || !seen) { free(inP); free(seen); return ORC_ENOMEM; }
    int32_t st[8] = {0};
    for (int t = 0; t < T; ++t)
        for (int r = 0; r < k; ++r) {
            int s = ids[(size_t)t * ld + r];
            if (s < 0 || s >= N) { free(inP); free(seen); return ORC_EINVAL; }
            if (!seen[s]) { seen[s] = 1; st[0]++; }
            if (r < kp && !inP[s]) { inP[s] = 1; st[1]++; }
        }
    for (int t = 0; t < T; ++t) {
        int32_t* id = ids + (size_t)t * ld;
        float* g = gates + (size_t)t * ld;
        for (int r = kp; r < k; ++r) {
            int s = id[r];
            if (inP[s]) continue;
            if (protect && protect[s]) { st[5]++; continue; }
            int best = -1;
            float bsim = 0.0f;
            for (int p = 0; p < N; ++p) {
                if (!inP[p]) continue;
                float v = sim[(size_t)s * N + p];
                if (best < 0 || v > bsim) { best = p; bsim = v; }
            }
            if (best >= 0 && bsim > rho) {
                int q = -1;
                for (int qq = 0; qq < k; ++qq)
                    if (id[qq] == best) q = qq;
                if (q >= 0) {
                    g[q] = g[q] + g[r];
                    id[r] = -1;
                    g[r] = 0.0f;
                    st[4]++;
                } else {
                    id[r] = best;
                    st[3]++;
                }
            } else {
                st[6]++;
            }
        }
    }
    memset(seen, 0, (size_t)N);
    for (int t = 0; t < T; ++t)
        for (int r = 0; r < k; ++r) {
            int s = ids[(size_t)t * ld + r];
            if (s >= 0 && !seen[s]) { seen[s] = 1; st[2]++; }
        }
    if (bitmap) {
        int words = (N + 31) / 32;
        for (int w = 0; w < words; ++w) bitmap[w] = 0u;
        for (int p = 0; p < N; ++p)
            if (inP[p]) bitmap[p / 32] |= 1u << (p % 32);
    }
    if (stats) memcpy(stats, st, sizeof st);
    free(inP);
    free(seen);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Capacity-bounded dispatch with weighted load.                       */
/* [MACS] 3.1 Eq. (2)-(3) (static capacity C = gamma |T| k / N),        */
/* 3.2 Eq. (6) (an expert's load is the sum of its tokens' weights w),  */
/* Fig. 1 / 3.4 (overflow tokens are rerouted locally, else dropped).   */
/*                                                                      */
/* Arithmetic: w_q = rint(w * 2^24) in int64 (exact, order-free sums);  */
/* S = sum_t w_q; C = floor(((double)S * k) * gamma / N) in double.     */
/* Phase 1, per expert: its (token, slot) pairs sorted by (gate desc,   */
/*   token asc); admitted = the longest prefix whose cumulative w_q     */
/*   stays <= C; the rest overflow.                                     */
/* Phase 2, rounds i = 0..R-k-1: every token with an overflowed slot    */
/*   proposes its lowest-rank overflowed slot to its rank-(k+i) expert, */
/*   carrying that slot's gate; each expert sorts its proposals by      */
/*   (gate desc, token asc) and admits the longest prefix with          */
/*   load + cumulative w_q <= C.                                        */
/* Slots still unplaced after the last round are dropped (gate lost).   */
/* Outputs: out_ids/out_gates [T][k] (dropped: -1, 0), status [T][k],   */
/* load[N] (final, in 2^-24 units), *cap = C.                           */
/* ------------------------------------------------------------------ */
typedef struct { float gate; int32_t token; int32_t slot; } orc_pair;

static int orc_pair_cmp(const void* a, const void* b) {
    const orc_pair* x = (const orc_pair*)a;
    const orc_pair* y = (const orc_pair*)b;
    if (x->gate > y->gate) return -1;
    if (x->gate < y->gate) return 1;
    return (x->token > y->token) - (x->token < y->token);
}

int64_t orc_fixed_weight(float w) { return (int64_t)rintf(w * 16777216.0f); }

int64_t orc_capacity_value(int64_t S, int k, float gamma, int N) {
    return (int64_t)floor(((double)S * (double)k) * (double)gamma / (double)N);
}

/* Per-expert capacity.  [MACS] 3.3 groups experts by modality (m_j = +1
 * visual, -1 text, 0 shared) and scales their capacity with the batch's
 * effective visual ratio R_v (Eq. 7); the page text stops before the
 * scaling formula.  Reading: C_j = floor(c * (1 + m_j * (R_v - 1/2))) with
 * c = ((double)S * k) * gamma / N the unfloored static capacity, so that
 * m_j = 0 (or R_v = 1/2) gives the static C and a modality's experts get up
 * to half as much again when the batch leans towards it.  Each operation
 * is rounded on its own, in this order. */
int64_t orc_capacity_expert(int64_t S, int k, float gamma, int N, int m, float r_v) {
    const double c = ((double)S * (double)k) * (double)gamma / (double)N;
    const double scale = 1.0 + (double)m * ((double)r_v - 0.5);
    return (int64_t)floor(c * scale);
}

int orc_capacity(const int32_t* ids, const float* gates, int ld, int T, int N, int k, int R,
                 const float* token_w, float gamma, int32_t* out_ids, float* out_gates,
                 uint8_t* status, int64_t* load, int64_t* cap, const int8_t* bias, float r_v) {
    if (!ids || !gates || !out_ids || !out_gates || !status || !load || T < 0 || N <= 0 || k <= 0 ||
        R < k || ld < R || !(gamma > 0.0f))
        return ORC_EINVAL;
    if (bias != NULL) {
        if (!(r_v >= 0.0f && r_v <= 1.0f)) return ORC_EINVAL;
        for (int e = 0; e < N; ++e)
            if (bias[e] < -1 || bias[e] > 1) return ORC_EINVAL;
    }
    int64_t* wq = (int64_t*)malloc(sizeof(int64_t) * (size_t)(T > 0 ? T : 1));
    orc_pair* buf = (orc_pair*)malloc(sizeof(orc_pair) * (size_t)(T > 0 ? T : 1));
    int32_t* pend = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
    if (!wq || !buf || !pend) { free(wq); free(buf); free(pend); return ORC_ENOMEM; }
    int64_t S = 0;
    for (int t = 0; t < T; ++t) {
        float w = token_w ? token_w[t] : 1.0f;
        if (!isfinite(w) || w < 0.0f) { free(wq); free(buf); free(pend); return ORC_EINVAL; }
        wq[t] = orc_fixed_weight(w);
        S += wq[t];
    }
    int64_t C = orc_capacity_value(S, k, gamma, N);
    if (cap) *cap = C;
    int64_t* Ce = (int64_t*)malloc(sizeof(int64_t) * (size_t)N);
    if (!Ce) { free(wq); free(buf); free(pend); return ORC_ENOMEM; }
    for (int e = 0; e < N; ++e) Ce[e] = bias ? orc_capacity_expert(S, k, gamma, N, bias[e], r_v) : C;
    const uint8_t PENDING = 255;
    for (int t = 0; t < T; ++t)
        for (int r = 0; r < k; ++r) {
            out_ids[(size_t)t * k + r] = ids[(size_t)t * ld + r];
            out_gates[(size_t)t * k + r] = gates[(size_t)t * ld + r];
            status[(size_t)t * k + r] = PENDING;
        }
    /* phase 1 */
    for (int e = 0; e < N; ++e) {
        int n = 0;
        for (int t = 0; t < T; ++t)
            for (int r = 0; r < k; ++r)
                if (ids[(size_t)t * ld + r] == e) {
                    buf[n].gate = gates[(size_t)t * ld + r];
                    buf[n].token = t;
                    buf[n].slot = r;
                    ++n;
                }
        qsort(buf, (size_t)n, sizeof(orc_pair), orc_pair_cmp);
        int64_t cum = 0;
        int open = 1;
        for (int i = 0; i < n; ++i) {
            int t = buf[i].token, r = buf[i].slot;
            if (open && cum + wq[t] <= Ce[e]) {
                cum += wq[t];
                status[(size_t)t * k + r] = ORC_SLOT_KEPT;
            } else {
                open = 0;
            }
        }
        load[e] = cum;
    }
    /* phase 2 */
    for (int i = 0; i + k < R; ++i) {
        for (int t = 0; t < T; ++t) {
            pend[t] = -1;
            for (int r = 0; r < k; ++r)
                if (status[(size_t)t * k + r] == PENDING) { pend[t] = r; break; }
        }
        for (int e = 0; e < N; ++e) {
            int n = 0;
            for (int t = 0; t < T; ++t)
                if (pend[t] >= 0 && ids[(size_t)t * ld + k + i] == e) {
                    buf[n].gate = gates[(size_t)t * ld + pend[t]];
                    buf[n].token = t;
                    buf[n].slot = pend[t];
                    ++n;
                }
            qsort(buf, (size_t)n, sizeof(orc_pair), orc_pair_cmp);
            int64_t cum = 0;
            int open = 1;
            for (int j = 0; j < n; ++j) {
                int t = buf[j].token, r = buf[j].slot;
                if (open && load[e] + cum + wq[t] <= Ce[e]) {
                    cum += wq[t];
                    status[(size_t)t * k + r] = ORC_SLOT_REROUTED;
                    out_ids[(size_t)t * k + r] = e;
                } else {
                    open = 0;
                }
            }
            load[e] += cum;
        }
    }
    for (int t = 0; t < T; ++t)
        for (int r = 0; r < k; ++r)
            if (status[(size_t)t * k + r] == PENDING) {
                status[(size_t)t * k + r] = ORC_SLOT_DROPPED;
                out_ids[(size_t)t * k + r] = -1;
                out_gates[(size_t)t * k + r] = 0.0f;
            }
    free(wq);
    free(buf);
    free(pend);
    free(Ce);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Expert-sorted permutation: the token sets I_j of [MACS] 3.1 as rows  */
/* ordered by (expert asc, token asc).  Slots with id -1 are skipped.   */
/* active[0] = number of experts with rows, active[1..] their ids asc.  */
/* ------------------------------------------------------------------ */
int orc_permute(const int32_t* ids, const float* gates, int ld, int T, int N, int k, int32_t* counts,
                int32_t* offsets, int32_t* row_token, float* row_gate, int32_t* active) {
    if (!ids || !gates || !counts || !offsets || T < 0 || N <= 0 || k <= 0 || ld < k) return ORC_EINVAL;
    for (int e = 0; e < N; ++e) counts[e] = 0;
    for (int t = 0; t < T; ++t)
        for (int r = 0; r < k; ++r) {
            int e = ids[(size_t)t * ld + r];
            if (e >= N) return ORC_EINVAL;
            if (e >= 0) counts[e]++;
        }
    offsets[0] = 0;
    for (int e = 0; e < N; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int na = 0;
    for (int e = 0; e < N; ++e) {
        int pos = offsets[e];
        for (int t = 0; t < T; ++t)
            for (int r = 0; r < k; ++r)
                if (ids[(size_t)t * ld + r] == e) {
                    if (row_token) row_token[pos] = t;
                    if (row_gate) row_gate[pos] = gates[(size_t)t * ld + r];
                    ++pos;
                }
        if (counts[e] > 0 && active) active[1 + na] = e;
        if (counts[e] > 0) ++na;
    }
    if (active) active[0] = na;
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Expert FFN and weighted combine, [MACS] 3.1 Eq. (1):                */
/*   y(x) = sum_{j in selected} g_j E_j(x),                            */
/*   E_j(x) = W_down_j ( silu(W_gate_j x) * (W_up_j x) ),               */
/*   silu(v) = v / (1 + exp(-v)).                                       */
/* All in double.  Weights: w_gate/w_up [N][I][H], w_down [N][H][I].    */
/* Computes y for the listed tokens only (tok[0..ntok)), y [ntok][H].   */
/* ------------------------------------------------------------------ */
int orc_ffn_combine(const void* x, int x_dtype, const void* w_gate, const void* w_up, const void* w_down,
                    int w_dtype, int T, int H, int I, int N, const int32_t* ids, const float* gates, int ld,
                    int k, const int32_t* tok, int ntok, double* y) {
    if (!x || !w_gate || !w_up || !w_down || !ids || !gates || !tok || !y || H <= 0 || I <= 0 || N <= 0 ||
        k <= 0 || ld < k || ntok < 0)
        return ORC_EINVAL;
    for (int n = 0; n < ntok; ++n) {
        int t = tok[n];
        if (t < 0 || t >= T) return ORC_EINVAL;
        for (int r = 0; r < k; ++r)
            if (ids[(size_t)t * ld + r] >= N) return ORC_EINVAL;
    }
    int rc = ORC_OK;
    /* tokens are independent: one thread computes a token's whole output row
       in the order below, so the result does not depend on the thread count */
#pragma omp parallel
    {
        double* xv = (double*)malloc(sizeof(double) * (size_t)H);
        double* act = (double*)malloc(sizeof(double) * (size_t)I);
        if (!xv || !act) {
#pragma omp atomic write
            rc = ORC_ENOMEM;
        }
#pragma omp for schedule(dynamic, 1)
        for (int n = 0; n < ntok; ++n) {
            if (!xv || !act) continue;
            int t = tok[n];
            for (int h = 0; h < H; ++h) xv[h] = ld_val(x, x_dtype, (size_t)t * H + h);
            double* yo = y + (size_t)n * H;
            for (int h = 0; h < H; ++h) yo[h] = 0.0;
            for (int r = 0; r < k; ++r) {
                int e = ids[(size_t)t * ld + r];
                if (e < 0) continue;
                double g = (double)gates[(size_t)t * ld + r];
                for (int i = 0; i < I; ++i) {
                    double a = 0.0, b = 0.0;
                    size_t base = ((size_t)e * I + i) * H;
                    for (int h = 0; h < H; ++h) {
                        a += ld_val(w_gate, w_dtype, base + h) * xv[h];
                        b += ld_val(w_up, w_dtype, base + h) * xv[h];
                    }
                    act[i] = a / (1.0 + exp(-a)) * b;
                }
                for (int h = 0; h < H; ++h) {
                    double acc = 0.0;
                    size_t base = ((size_t)e * H + h) * I;
                    for (int i = 0; i < I; ++i) acc += ld_val(w_down, w_dtype, base + i) * act[i];
                    yo[h] += g * acc;
                }
            }
        }
        free(xv);
        free(act);
    }
    return rc;
}

/* ------------------------------------------------------------------ */
/* Entropy-weighted token load.  [MACS] 3.2 Eqs. (4)-(5), 3.3 Eq. (7).   */
/*                                                                      */
/* For every token t, its feature vector z (the layer's input row,      */
/* D = H values) gives p = Softmax(z) and the Shannon entropy           */
/*   H(t) = -sum_d p_d ln p_d = ln Z - (sum_d e_d (z_d - m)) / Z,        */
/* with m = max z, e_d = exp(z_d - m), Z = sum e_d.  Over the batch's   */
/* visual tokens: mu = mean H, sigma = population standard deviation    */
/* (Eq. 4's batch statistics), Htilde = (H - mu) / (sigma + eps).        */
/* Weights (Eq. 5): w = sigmoid(-delta * Htilde) for visual tokens, 1    */
/* for text tokens.  Effective visual ratio (Eq. 7):                     */
/*   R_v = sum_{visual} w / sum_{all} w  (0 for an empty batch).         */
/* Everything in double.  The entropy is computed for every token; only */
/* the visual ones enter the statistics.                                */
/* ------------------------------------------------------------------ */
int orc_token_weights(const void* x, int x_dtype, int T, int H, const uint8_t* is_visual, double delta, double eps,
                      double* entropy, double* w, double* r_v) {
    if (T < 0 || H < 1 || (T > 0 && (x == NULL || is_visual == NULL || entropy == NULL || w == NULL)))
        return ORC_EINVAL;
    for (int t = 0; t < T; ++t) {
        double m = -INFINITY;
        for (int d = 0; d < H; ++d) {
            const double z = ld_val(x, x_dtype, (size_t)t * H + d);
            if (z > m) m = z;
        }
        double Z = 0.0, S1 = 0.0;
        for (int d = 0; d < H; ++d) {
            const double z = ld_val(x, x_dtype, (size_t)t * H + d) - m;
            const double e = exp(z);
            Z += e;
            S1 += e * z;
        }
        entropy[t] = log(Z) - S1 / Z;
    }
    int nv = 0;
    double sum = 0.0;
    for (int t = 0; t < T; ++t)
        if (is_visual[t]) {
            ++nv;
            sum += entropy[t];
        }
    const double mu = nv > 0 ? sum / nv : 0.0;
    double var = 0.0;
    for (int t = 0; t < T; ++t)
        if (is_visual[t]) var += (entropy[t] - mu) * (entropy[t] - mu);
    const double sigma = nv > 0 ? sqrt(var / nv) : 0.0;
    double wv = 0.0, wall = 0.0;
    for (int t = 0; t < T; ++t) {
        if (is_visual[t]) {
            const double ht = (entropy[t] - mu) / (sigma + eps);
            w[t] = 1.0 / (1.0 + exp(delta * ht));
            wv += w[t];
        } else {
            w[t] = 1.0;
        }
        wall += w[t];
    }
    if (r_v != NULL) *r_v = wall > 0.0 ? wv / wall : 0.0;
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Expert similarity from calibration tokens.  [SERE] 4.2: the          */
/* similarity matrix is computed offline as the Frobenius similarity    */
/* of the experts' outputs on calibration data:                         */
/*   sim[i][j] = <E_i(X), E_j(X)>_F / (||E_i(X)||_F ||E_j(X)||_F)        */
/* with E_e(X) the [n][H] matrix of expert e's SwiGLU outputs on the n   */
/* calibration tokens ([MACS] Eq. 1's E_j).  Everything in double.      */
/* Reading: the diagonal is 1, and a pair involving an expert whose      */
/* output is all zero has similarity 0.                                  */
/* ------------------------------------------------------------------ */
int orc_similarity(const void* x, int x_dtype, int n, int H, const void* w_gate, const void* w_up,
                   const void* w_down, int w_dtype, int I, int N, double* sim) {
    if (n < 1 || H < 1 || I < 1 || N < 1 || !x || !w_gate || !w_up || !w_down || !sim) return ORC_EINVAL;
    double* E = (double*)malloc(sizeof(double) * (size_t)N * n * H);
    if (!E) return ORC_ENOMEM;
    int rc = ORC_OK;
    /* experts are independent: one thread computes an expert's outputs for
       every calibration token, in the order below */
#pragma omp parallel
    {
        double* xv = (double*)malloc(sizeof(double) * (size_t)H);
        double* act = (double*)malloc(sizeof(double) * (size_t)I);
        if (!xv || !act) {
#pragma omp atomic write
            rc = ORC_ENOMEM;
        }
#pragma omp for schedule(dynamic, 1)
        for (int e = 0; e < N; ++e) {
            if (!xv || !act) continue;
            for (int t = 0; t < n; ++t) {
                for (int h = 0; h < H; ++h) xv[h] = ld_val(x, x_dtype, (size_t)t * H + h);
                for (int i = 0; i < I; ++i) {
                    double a = 0.0, b = 0.0;
                    const size_t base = ((size_t)e * I + i) * H;
                    for (int h = 0; h < H; ++h) {
                        a += ld_val(w_gate, w_dtype, base + h) * xv[h];
                        b += ld_val(w_up, w_dtype, base + h) * xv[h];
                    }
                    act[i] = a / (1.0 + exp(-a)) * b;
                }
                double* eo = E + ((size_t)e * n + t) * H;
                for (int h = 0; h < H; ++h) {
                    double acc = 0.0;
                    const size_t base = ((size_t)e * H + h) * I;
                    for (int i = 0; i < I; ++i) acc += ld_val(w_down, w_dtype, base + i) * act[i];
                    eo[h] = acc;
                }
            }
        }
        free(xv);
        free(act);
    }
    if (rc != ORC_OK) { free(E); return rc; }
    const size_t K = (size_t)n * H;
    /* each pair (i, j) is summed by one thread in the order below */
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < N; ++i)
        for (int j = i; j < N; ++j) {
            double gij = 0.0, gii = 0.0, gjj = 0.0;
            const double* a = E + (size_t)i * K;
            const double* b = E + (size_t)j * K;
            for (size_t q = 0; q < K; ++q) {
                gij += a[q] * b[q];
                gii += a[q] * a[q];
                gjj += b[q] * b[q];
            }
            double v = (i == j) ? 1.0 : ((gii > 0.0 && gjj > 0.0) ? gij / sqrt(gii * gjj) : 0.0);
            sim[(size_t)i * N + j] = v;
            sim[(size_t)j * N + i] = v;
        }
    free(E);
    return ORC_OK;
}
