/*
 * spec_verify_oracle.c -- plain float64 CPU oracle of the batched
 * speculative-sampling verifier.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test-suite, the smoke
 * check and the CPU-baseline leg of the benchmark load this file.  It shares
 * no source, header, table or helper with the CUDA library; the two sides
 * agree only on the published definitions they both restate.
 *
 * Sources restated here (web pages, cited by title and section):
 *   [P1] "深入推测解码：从概念到实现" (translation of M. Abboud, "Exploring
 *        Speculative Decoding: From Concept to Implementation"),
 *        sections 伪代码 (pseudocode) and 保证原始分布 (guaranteeing the
 *        original distribution, steps 1-4 and the q=0.4 / p=0.2 example).
 *   [P2] "RTP-LLM Speculative Engine 深度解析", section 拒绝采样算法
 *        (SpeculativeSampler::stochasticSample).
 *   [P3] "投机采样" (razer666.cn), sections 第三步 / 第四步 / 第五步 of
 *        投机解码算法, the output-length cases after 第五步, and
 *        验收标准 / 精确匹配 (exact-match acceptance).
 *   [Philox] J. Salmon, M. Moraes, R. Dror, D. Shaw, "Parallel Random
 *        Numbers: As Easy as 1, 2, 3", SC'11 -- Philox4x32 with 10 rounds.
 *
 * What it computes, per request b (requests are independent):
 *   p_j = softmax(l_j / T_b) for sampling requests (T_b > 0), in float64,
 *   summed sequentially x = 0..V-1.  For j = 0..n_b-1, in order:
 *     sampling: accept draft x_j iff p_j(x_j) > 0 and
 *               (q_j(x_j) == 0 or u_j <= p_j(x_j) / q_j(x_j));
 *     greedy (T_b == 0): accept iff x_j == argmax l_j (lowest index).
 *   Stop at the first rejection j: emit a token from
 *     norm(max(0, p_j - q_j)) by inverse CDF with u'_j (sampling), or
 *     argmax l_j (greedy).
 *   If all n_b drafts are accepted: emit the bonus token from p_{n_b}
 *   (sampling, inverse CDF with u'_{n_b}) or argmax l_{n_b} (greedy).
 *   out_ids[b] = accepted drafts, the emitted token, then -1 padding;
 *   out_num_accepted[b] = number of accepted drafts.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - uniforms: u = ((x >> 8) + 1) * 2^-24 in (0, 1] from a Philox4x32-10
 *     block with key (seed lo, seed hi) and counter (b, j, 0, 0); lane 0 is
 *     the acceptance uniform of row j, lane 1 the emission uniform of row j;
 *   - inverse CDF: the smallest x with C(x) >= u' * C(V-1), where C is the
 *     sequential prefix sum of the (unnormalised) weights;
 *   - q is used as given (not renormalised); q(x_j) == 0 with p(x_j) > 0
 *     accepts; a residual with zero total mass falls back to p;
 *   - bad requests (num_draft outside [0, K], temperature NaN / negative /
 *     infinite, a draft id outside [0, V), or a sampling row whose logits are
 *     all -inf) get out_ids = -1 and out_num_accepted = -1.
 *
 * Typical acceptance ([P3] 验收标准, "Typical Acceptance": a draft is accepted
 * when its probability under the target exceeds a hard threshold, and the
 * longest such prefix is kept) is the lossy alternative rule, selected by
 * mode ORACLE_TYPICAL: accept x_j iff p_j(x_j) > 0 and p_j(x_j) >= threshold;
 * the token after the kept prefix (whether a draft was refused or all were
 * kept) is drawn from p at that row by the same inverse CDF with u'.  q is not
 * used.  Greedy requests are verified by exact match in either mode.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------- */
/* Philox4x32-10 [Philox], written from the paper's definition.            */
/* ---------------------------------------------------------------------- */

static const uint32_t PHILOX_MUL0 = 0xD2511F53u;
static const uint32_t PHILOX_MUL1 = 0xCD9E8D57u;
static const uint32_t PHILOX_WEYL0 = 0x9E3779B9u; /* golden ratio */
static const uint32_t PHILOX_WEYL1 = 0xBB67AE85u; /* sqrt(3) - 1 */

void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                          uint32_t out[4]) {
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { /* the key schedule adds the Weyl constants */
            k0 += PHILOX_WEYL0;
            k1 += PHILOX_WEYL1;
        }
        uint64_t prod0 = (uint64_t)PHILOX_MUL0 * (uint64_t)c0;
        uint64_t prod1 = (uint64_t)PHILOX_MUL1 * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* 32 random bits -> uniform in (0, 1]: ((x >> 8) + 1) * 2^-24. */
double oracle_uniform_from_bits(uint32_t x) {
    return (double)((x >> 8) + 1u) * (1.0 / 16777216.0);
}

/* The two uniforms of row j of request b: lane 0 (acceptance), lane 1
 * (emission), from the block with key (seed lo, seed hi), counter (b, j, 0, 0). */
void oracle_row_uniforms(uint64_t seed, uint64_t b, uint32_t j, double* u_accept,
                         double* u_emit) {
    uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
    uint32_t ctr[4] = {(uint32_t)b, j, 0u, 0u};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    *u_accept = oracle_uniform_from_bits(out[0]);
    *u_emit = oracle_uniform_from_bits(out[1]);
}

/* ---------------------------------------------------------------------- */
/* Inputs, converted exactly to float64.                                   */
/* ---------------------------------------------------------------------- */

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };
enum { ORACLE_LOSSLESS = 0, ORACLE_TYPICAL = 1 };

static double logit_at(const void* logits, int dtype, size_t idx) {
    if (dtype == ORACLE_BF16) {
        uint16_t h = ((const uint16_t*)logits)[idx];
        uint32_t bits = (uint32_t)h << 16; /* bf16 is the top half of an f32 */
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float*)logits)[idx];
}

/* Row (b, j) of target_logits [B, K+1, V] into dst[V] (float64). */
static void load_logit_row(const void* logits, int dtype, int K, int V, int b, int j,
                           double* dst) {
    size_t base = ((size_t)b * (size_t)(K + 1) + (size_t)j) * (size_t)V;
    for (int x = 0; x < V; ++x) dst[x] = logit_at(logits, dtype, base + (size_t)x);
}

/* ---------------------------------------------------------------------- */
/* The method's steps.                                                     */
/* ---------------------------------------------------------------------- */

/* Greedy target token: the lowest index among the maxima of the raw logits
 * ([P3] 验收标准 / 精确匹配: the token of maximum probability; softmax is
 * monotone, so the raw logits decide). */
static int argmax_lowest(const double* l, int V) {
    int best = 0;
    for (int x = 1; x < V; ++x)
        if (l[x] > l[best]) best = x;
    return best;
}

/* p = softmax(l / T) in float64: M = max_x l(x)/T, Z = sum_x exp(l(x)/T - M)
 * summed sequentially, p(x) = exp(l(x)/T - M) / Z.  Returns Z (0 when the
 * row has no finite logit). */
static double softmax_t(const double* l, int V, double T, double* p) {
    double M = -INFINITY;
    for (int x = 0; x < V; ++x) {
        double s = l[x] / T;
        if (s > M) M = s;
    }
    if (M == -INFINITY) return 0.0;
    double Z = 0.0;
    for (int x = 0; x < V; ++x) {
        p[x] = exp(l[x] / T - M);
        Z += p[x];
    }
    for (int x = 0; x < V; ++x) p[x] /= Z;
    return Z;
}

/* Inverse CDF over non-negative weights w[V]: C(x) = sum_{y<=x} w(y) summed
 * sequentially, S = C(V-1); returns the smallest x with C(x) >= u * S, and the
 * normalised interval (C(x-1)/S, C(x)/S] of the chosen x.  If probe >= 0 the
 * interval of x = probe is returned in probe_lo/probe_hi as well. */
static int inverse_cdf(const double* w, int V, double u, double* S_out, double* lo_out,
                       double* hi_out, int probe, double* probe_lo, double* probe_hi) {
    double S = 0.0;
    for (int x = 0; x < V; ++x) S += w[x];
    double t = u * S;
    double C = 0.0;
    int pick = -1;
    for (int x = 0; x < V; ++x) {
        double before = C;
        C += w[x];
        if (pick < 0 && C >= t) {
            pick = x;
            *lo_out = before / S;
            *hi_out = C / S;
        }
        if (x == probe) {
            *probe_lo = before / S;
            *probe_hi = C / S;
        }
    }
    if (pick < 0) { /* unreachable for u <= 1: C(V-1) == S >= t */
        pick = V - 1;
        *lo_out = *hi_out = 1.0;
    }
    *S_out = S;
    return pick;
}

/* Per-row diagnostics (ORACLE_ROW_W doubles per (b, j)). */
enum {
    R_PX = 0,     /* p_j(x_j) (sampling rows j < n_b that were tested) */
    R_QX = 1,     /* q_j(x_j) */
    R_U = 2,      /* acceptance uniform u_j */
    R_ACCEPT = 3, /* 1 accepted, 0 rejected, -1 not tested */
    ORACLE_ROW_W = 4
};
/* Per-request diagnostics (ORACLE_REQ_W doubles per b). */
enum {
    Q_MODE = 0,   /* -1 bad, 0 greedy, 1 residual, 2 bonus, 3 residual->p fallback,
                     4 typical acceptance: drawn from p at the row after the kept prefix */
    Q_NACC = 1,   /* number of accepted drafts */
    Q_EROW = 2,   /* row the emitted token came from */
    Q_UEMIT = 3,  /* emission uniform u' (sampling) */
    Q_MASS = 4,   /* total mass of the emission weights (sum r, or sum p) */
    Q_LO = 5,     /* normalised CDF before the emitted token */
    Q_HI = 6,     /* normalised CDF at the emitted token */
    Q_PLO = 7,    /* same two for the probe token, if one was given */
    Q_PHI = 8,
    ORACLE_REQ_W = 9
};

/* One request.  u_accept[j], u_emit[j] for j = 0..K are its uniforms.
 * p, r: scratch of V doubles.  Returns 0, or -1 for a bad request. */
static int verify_request(const void* logits, int dtype, const float* draft_probs,
                          const int32_t* draft_ids, int n, float temperature, int b, int K,
                          int V, const double* u_accept, const double* u_emit,
                          int32_t* out_ids, int32_t* out_nacc, double* row_diag,
                          double* req_diag, int probe, double* l, double* p, double* r,
                          int rule, double threshold) {
    for (int j = 0; j <= K; ++j) out_ids[j] = -1;
    *out_nacc = -1;
    if (req_diag) {
        for (int i = 0; i < ORACLE_REQ_W; ++i) req_diag[i] = NAN;
        req_diag[Q_MODE] = -1;
    }
    if (row_diag)
        for (int j = 0; j <= K; ++j) {
            for (int i = 0; i < ORACLE_ROW_W; ++i) row_diag[j * ORACLE_ROW_W + i] = NAN;
            row_diag[j * ORACLE_ROW_W + R_ACCEPT] = -1;
        }

    /* validation (bad requests produce -1 everywhere) */
    if (n < 0 || n > K) return -1;
    double T = (double)temperature;
    if (!(T >= 0.0) || isinf(T)) return -1; /* NaN, negative or infinite */
    for (int j = 0; j < n; ++j)
        if (draft_ids[j] < 0 || draft_ids[j] >= V) return -1;
    const int greedy = (T == 0.0);
    if (!greedy) {
        for (int j = 0; j <= n; ++j) { /* every row the method may need */
            load_logit_row(logits, dtype, K, V, b, j, l);
            int finite = 0;
            for (int x = 0; x < V && !finite; ++x) finite = (l[x] != -INFINITY);
            if (!finite) return -1;
        }
    }

    int accepted = 0, emitted = -1, mode = greedy ? 0 : 2, erow = n;
    double lo = NAN, hi = NAN, mass = NAN, plo = NAN, phi = NAN;

    /* [P3] 第三步: test the drafts in order; [P2] 拒绝采样算法: break at the
     * first rejection. */
    for (int j = 0; j < n; ++j) {
        const int xj = draft_ids[j];
        load_logit_row(logits, dtype, K, V, b, j, l);
        if (greedy) {
            int g = argmax_lowest(l, V);
            if (row_diag) row_diag[j * ORACLE_ROW_W + R_ACCEPT] = (g == xj);
            if (g == xj) {
                ++accepted;
                continue;
            }
            emitted = g; /* the target's own token replaces the mismatch */
            erow = j;
            break;
        }
        softmax_t(l, V, T, p);
        const double px = p[xj];
        if (rule == ORACLE_TYPICAL) {
            /* [P3] 验收标准, Typical Acceptance: a hard threshold on p(x_j) */
            const int accept = (px > 0.0) && (px >= threshold);
            if (row_diag) {
                row_diag[j * ORACLE_ROW_W + R_PX] = px;
                row_diag[j * ORACLE_ROW_W + R_ACCEPT] = accept;
            }
            if (accept) {
                ++accepted;
                continue;
            }
            erow = j;  /* the target's own token at the first refused position */
            mode = 4;
            emitted = inverse_cdf(p, V, u_emit[j], &mass, &lo, &hi, probe, &plo, &phi);
            break;
        }
        const float* q = draft_probs + ((size_t)b * (size_t)K + (size_t)j) * (size_t)V;
        const double qx = (double)q[xj];
        const double u = u_accept[j];
        /* [P1] 保证原始分布 step 3: accept with probability min(1, p/q) */
        const int accept = (px > 0.0) && (qx == 0.0 || u <= px / qx);
        if (row_diag) {
            row_diag[j * ORACLE_ROW_W + R_PX] = px;
            row_diag[j * ORACLE_ROW_W + R_QX] = qx;
            row_diag[j * ORACLE_ROW_W + R_U] = u;
            row_diag[j * ORACLE_ROW_W + R_ACCEPT] = accept;
        }
        if (accept) {
            ++accepted;
            continue;
        }
        /* [P1] step 4, [P3] 第四步: resample from norm(max(0, p - q)) */
        for (int x = 0; x < V; ++x) {
            double d = p[x] - (double)q[x];
            r[x] = d > 0.0 ? d : 0.0;
        }
        double S = 0.0;
        for (int x = 0; x < V; ++x) S += r[x];
        erow = j;
        if (S > 0.0) {
            mode = 1;
            emitted = inverse_cdf(r, V, u_emit[j], &mass, &lo, &hi, probe, &plo, &phi);
        } else { /* zero residual mass (only with unnormalised q): sample p */
            mode = 3;
            emitted = inverse_cdf(p, V, u_emit[j], &mass, &lo, &hi, probe, &plo, &phi);
        }
        break;
    }

    if (accepted == n) {
        /* [P3] 第五步 and the third output-length case: all drafts accepted,
         * one more token from the target's distribution at position n. */
        load_logit_row(logits, dtype, K, V, b, n, l);
        erow = n;
        if (greedy) {
            emitted = argmax_lowest(l, V);
        } else {
            mode = rule == ORACLE_TYPICAL ? 4 : 2;
            softmax_t(l, V, T, p);
            emitted = inverse_cdf(p, V, u_emit[n], &mass, &lo, &hi, probe, &plo, &phi);
        }
    }

    for (int j = 0; j < accepted; ++j) out_ids[j] = draft_ids[j];
    out_ids[accepted] = emitted;
    *out_nacc = accepted;
    if (req_diag) {
        req_diag[Q_MODE] = mode;
        req_diag[Q_NACC] = accepted;
        req_diag[Q_EROW] = erow;
        req_diag[Q_UEMIT] = greedy ? NAN : u_emit[erow];
        req_diag[Q_MASS] = mass;
        req_diag[Q_LO] = lo;
        req_diag[Q_HI] = hi;
        req_diag[Q_PLO] = plo;
        req_diag[Q_PHI] = phi;
    }
    return 0;
}

/*
 * The oracle over a batch.
 *   target_logits [B, K+1, V] (dtype 0 = f32, 1 = bf16 bit patterns),
 *   draft_probs [B, K, V] f32 (may be NULL if every request is greedy),
 *   draft_ids [B, K], num_draft [B], temperature [B].
 *   uniforms: NULL -> Philox(seed, req_index[b] (or b), j); else [B, K+1, 2]
 *             doubles (lane 0 acceptance, lane 1 emission) used as given.
 *   req_index: NULL -> b; else the global request index used as the Philox
 *              counter of local request b.
 *   probe: NULL, or [B] token ids whose emission-CDF interval is reported.
 *   out_ids [B, K+1], out_num_accepted [B]; row_diag [B, K+1, ORACLE_ROW_W]
 *   and req_diag [B, ORACLE_REQ_W] may be NULL.
 *   n_threads <= 0: the OpenMP default.
 * Returns the number of bad requests, or -1 on an argument error.
 */
int oracle_spec_verify_rule(const void* target_logits, int logits_dtype,
                            const float* draft_probs, const int32_t* draft_ids,
                            const int32_t* num_draft, const float* temperature, uint64_t seed,
                            int B, int K, int V, const int64_t* req_index,
                            const double* uniforms, const int32_t* probe, int32_t* out_ids,
                            int32_t* out_num_accepted, double* row_diag, double* req_diag,
                            int n_threads, int rule, double threshold) {
    if (rule != ORACLE_LOSSLESS && rule != ORACLE_TYPICAL) return -1;
    if (B < 0 || K < 0 || K > 63 || V <= 0 || !target_logits || !draft_ids || !num_draft ||
        !temperature || !out_ids || !out_num_accepted)
        return -1;
    if (logits_dtype != ORACLE_F32 && logits_dtype != ORACLE_BF16) return -1;
    int bad = 0;
#ifdef _OPENMP
    if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads) reduction(+ : bad)
#endif
    {
        double* scratch = (double*)malloc(sizeof(double) * 3 * (size_t)V);
        double *l = scratch, *p = scratch + V, *r = scratch + 2 * (size_t)V;
        double ua[64], ue[64]; /* K + 1 <= 64 */
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int b = 0; b < B; ++b) {
            const uint64_t gb = req_index ? (uint64_t)req_index[b] : (uint64_t)b;
            for (int j = 0; j <= K; ++j) {
                if (uniforms) {
                    ua[j] = uniforms[((size_t)b * (size_t)(K + 1) + (size_t)j) * 2 + 0];
                    ue[j] = uniforms[((size_t)b * (size_t)(K + 1) + (size_t)j) * 2 + 1];
                } else {
                    oracle_row_uniforms(seed, gb, (uint32_t)j, &ua[j], &ue[j]);
                }
            }
            int rc = -1;
            if (draft_probs != NULL || temperature[b] == 0.0f || num_draft[b] == 0 ||
                rule == ORACLE_TYPICAL) {
                /* greedy requests, requests without drafts and the typical rule
                   read no q */
                rc = verify_request(target_logits, logits_dtype, draft_probs,
                                    draft_ids + (size_t)b * (size_t)K, num_draft[b],
                                    temperature[b], b, K, V, ua, ue,
                                    out_ids + (size_t)b * (size_t)(K + 1), &out_num_accepted[b],
                                    row_diag ? row_diag + (size_t)b * (size_t)(K + 1) * ORACLE_ROW_W : NULL,
                                    req_diag ? req_diag + (size_t)b * ORACLE_REQ_W : NULL,
                                    probe ? probe[b] : -1, l, p, r, rule, threshold);
            } else {
                for (int j = 0; j <= K; ++j) out_ids[(size_t)b * (size_t)(K + 1) + j] = -1;
                out_num_accepted[b] = -1;
            }
            if (rc != 0) ++bad;
        }
        free(scratch);
    }
    return bad;
}

/* The lossless rule (the method of the pages). */
int oracle_spec_verify(const void* target_logits, int logits_dtype, const float* draft_probs,
                       const int32_t* draft_ids, const int32_t* num_draft,
                       const float* temperature, uint64_t seed, int B, int K, int V,
                       const int64_t* req_index, const double* uniforms, const int32_t* probe,
                       int32_t* out_ids, int32_t* out_num_accepted, double* row_diag,
                       double* req_diag, int n_threads) {
    return oracle_spec_verify_rule(target_logits, logits_dtype, draft_probs, draft_ids,
                                   num_draft, temperature, seed, B, K, V, req_index, uniforms,
                                   probe, out_ids, out_num_accepted, row_diag, req_diag,
                                   n_threads, ORACLE_LOSSLESS, 0.0);
}

/* ---------------------------------------------------------------------- */
/* Token-tree verification.                                                */
/* ---------------------------------------------------------------------- */

/* Row v of a [B, N, V] logits array into dst[V] (float64). */
static void load_node_row(const void* logits, int dtype, int N, int V, int b, int v,
                          double* dst) {
    size_t base = ((size_t)b * (size_t)N + (size_t)v) * (size_t)V;
    for (int x = 0; x < V; ++x) dst[x] = logit_at(logits, dtype, base + (size_t)x);
}

/*
 * One request of token-tree verification ([P3] 验证方案: the candidate
 * sequences share prefixes in a trie, and the target scores every node in one
 * pass; the verifier walks the trie from the root).  Node 0 is the root (the
 * accepted context); node c >= 1 carries token tok[c] and parent par[c] < c.
 * Row v of the logits is the target's distribution of the token after node
 * v's prefix; row c of q the draft distribution tok[c] was drawn from.
 *   greedy (T == 0, [P3] 精确匹配): at node v, the first child (in index
 *     order) whose token is the argmax of row v is accepted; else the argmax
 *     is emitted.
 *   sampling: the children of v are tested in index order against a running
 *     target r (r = p_v first): child c is accepted with probability
 *     min(1, r(x)/q_c(x)); after a rejection r becomes
 *     norm(max(0, r - q_c)) (kept as it was if that has no mass).  When no
 *     child is accepted the token is drawn from the last residual (from r if
 *     it had no mass, from p_v at a node without children).
 * ua[c] is the acceptance uniform of child c, ue[v] the emission uniform of
 * node v.  out[0..a-1] are the tokens of the accepted path, out[a] the
 * emitted token.  Returns 0, or -1 for a bad request.
 */
static int verify_tree_request(const void* logits, int dtype, const float* draft_probs,
                               const int32_t* tok, const int32_t* par, int n, float temperature,
                               int b, int N, int V, const double* ua, const double* ue,
                               int32_t* out, int32_t* out_nacc, int32_t* out_last,
                               double* node_diag, double* req_diag, int probe, double* l,
                               double* r, double* w) {
    for (int c = 0; c < N; ++c) out[c] = -1;
    *out_nacc = -1;
    *out_last = -1;
    if (node_diag)
        for (int c = 0; c < N; ++c) {
            for (int k = 0; k < ORACLE_ROW_W; ++k) node_diag[c * ORACLE_ROW_W + k] = NAN;
            node_diag[c * ORACLE_ROW_W + R_ACCEPT] = -1;
        }
    if (req_diag) {
        for (int k = 0; k < ORACLE_REQ_W; ++k) req_diag[k] = NAN;
        req_diag[Q_MODE] = -1;
    }
    const double T = (double)temperature;
    if (n < 1 || n > N) return -1;
    if (isnan(T) || T < 0.0 || isinf(T)) return -1;
    for (int c = 1; c < n; ++c) {
        if (par[c] < 0 || par[c] >= c) return -1;
        if (tok[c] < 0 || tok[c] >= V) return -1;
    }
    const int greedy = (T == 0.0);
    if (!greedy) {
        if (n > 1 && draft_probs == NULL) return -1;
        for (int v = 0; v < n; ++v) { /* every node row needs a finite logit */
            load_node_row(logits, dtype, N, V, b, v, l);
            int finite = 0;
            for (int x = 0; x < V; ++x)
                if (l[x] > -INFINITY) finite = 1;
            if (finite == 0) return -1;
        }
    }

    int v = 0, depth = 0, emitted = -1, mode = greedy ? 0 : 2;
    double mass = NAN, lo = NAN, hi = NAN, plo = NAN, phi = NAN;
    for (;;) {
        load_node_row(logits, dtype, N, V, b, v, l);
        if (greedy) {
            const int g = argmax_lowest(l, V);
            int next = -1;
            for (int c = v + 1; c < n && next < 0; ++c)
                if (par[c] == v) {
                    if (node_diag) node_diag[c * ORACLE_ROW_W + R_ACCEPT] = tok[c] == g;
                    if (tok[c] == g) next = c;
                }
            if (next < 0) {
                emitted = g;
                break;
            }
            out[depth++] = tok[next];
            v = next;
            continue;
        }
        softmax_t(l, V, T, r); /* the running target starts at p_v */
        const double* emit_w = r;
        int has_child = 0, next = -1;
        mode = 2;
        for (int c = v + 1; c < n; ++c) {
            if (par[c] != v) continue;
            has_child = 1;
            const float* q = draft_probs + ((size_t)b * (size_t)N + (size_t)c) * (size_t)V;
            const int x = tok[c];
            const double rx = r[x], qx = (double)q[x], u = ua[c];
            const int accept = (rx > 0.0) && (qx == 0.0 || u <= rx / qx);
            if (node_diag) {
                node_diag[c * ORACLE_ROW_W + R_PX] = rx;
                node_diag[c * ORACLE_ROW_W + R_QX] = qx;
                node_diag[c * ORACLE_ROW_W + R_U] = u;
                node_diag[c * ORACLE_ROW_W + R_ACCEPT] = accept;
            }
            if (accept) {
                next = c;
                break;
            }
            /* rejected: the residual max(0, r - q_c) */
            double S = 0.0;
            for (int y = 0; y < V; ++y) {
                const double e = r[y] - (double)q[y];
                w[y] = e > 0.0 ? e : 0.0;
                S += w[y];
            }
            if (S > 0.0) {
                emit_w = w; /* unnormalised: the inverse CDF normalises */
                mode = 1;
                int more = 0; /* a later sibling tests against the normalised residual */
                for (int c2 = c + 1; c2 < n; ++c2)
                    if (par[c2] == v) more = 1;
                if (more)
                    for (int y = 0; y < V; ++y) r[y] = w[y] / S;
            } else {
                emit_w = r; /* no residual mass: r stays */
                mode = 3;
            }
        }
        if (next >= 0) {
            out[depth++] = tok[next];
            v = next;
            continue;
        }
        if (!has_child) mode = 2;
        emitted = inverse_cdf(emit_w, V, ue[v], &mass, &lo, &hi, probe, &plo, &phi);
        break;
    }
    out[depth] = emitted;
    *out_nacc = depth;
    *out_last = v;
    if (req_diag) {
        req_diag[Q_MODE] = mode;
        req_diag[Q_NACC] = depth;
        req_diag[Q_EROW] = v;
        req_diag[Q_UEMIT] = greedy ? NAN : ue[v];
        req_diag[Q_MASS] = mass;
        req_diag[Q_LO] = lo;
        req_diag[Q_HI] = hi;
        req_diag[Q_PLO] = plo;
        req_diag[Q_PHI] = phi;
    }
    return 0;
}

/*
 * Token-tree verification over a batch.
 *   target_logits [B, N, V]; draft_probs [B, N, V] f32 (row 0 unused; may be
 *   NULL if no sampling request has a child); tree_tokens [B, N] and
 *   tree_parents [B, N] (entries of node 0 unused); num_nodes [B] in [1, N];
 *   temperature [B].
 *   uniforms: NULL -> Philox(seed, req_index[b] (or b), ...): child c's
 *             acceptance uniform is lane 0 of block (b, c - 1), node v's
 *             emission uniform lane 1 of block (b, v); else [B, N, 2] doubles
 *             (lane 0 of entry c - 1 for child c, lane 1 of entry v for v).
 *   out_ids [B, N], out_num_accepted [B], out_last_node [B]; node_diag
 *   [B, N, ORACLE_ROW_W] (per child c: r(x), q_c(x), u, accepted) and req_diag
 *   [B, ORACLE_REQ_W] may be NULL.
 * Returns the number of bad requests, or -1 on an argument error.
 */
int oracle_tree_verify(const void* target_logits, int logits_dtype, const float* draft_probs,
                       const int32_t* tree_tokens, const int32_t* tree_parents,
                       const int32_t* num_nodes, const float* temperature, uint64_t seed, int B,
                       int N, int V, const int64_t* req_index, const double* uniforms,
                       const int32_t* probe, int32_t* out_ids, int32_t* out_num_accepted,
                       int32_t* out_last_node, double* node_diag, double* req_diag,
                       int n_threads) {
    if (B < 0 || N < 1 || N > 64 || V <= 0 || !target_logits || !tree_tokens ||
        !tree_parents || !num_nodes || !temperature || !out_ids || !out_num_accepted ||
        !out_last_node)
        return -1;
    if (logits_dtype != ORACLE_F32 && logits_dtype != ORACLE_BF16) return -1;
    int bad = 0;
#ifdef _OPENMP
    if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads) reduction(+ : bad)
#endif
    {
        double* scratch = (double*)malloc(sizeof(double) * 3 * (size_t)V);
        double *l = scratch, *r = scratch + V, *w = scratch + 2 * (size_t)V;
        double ua[64], ue[64];
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int b = 0; b < B; ++b) {
            const uint64_t gb = req_index ? (uint64_t)req_index[b] : (uint64_t)b;
            for (int v = 0; v < N; ++v) {
                double a0, e0;
                if (uniforms) {
                    a0 = uniforms[((size_t)b * (size_t)N + (size_t)v) * 2 + 0];
                    e0 = uniforms[((size_t)b * (size_t)N + (size_t)v) * 2 + 1];
                } else {
                    oracle_row_uniforms(seed, gb, (uint32_t)v, &a0, &e0);
                }
                ue[v] = e0;
                if (v + 1 < 64) ua[v + 1] = a0; /* block (b, v) lane 0 -> child v + 1 */
            }
            ua[0] = NAN;
            const int rc = verify_tree_request(
                target_logits, logits_dtype, draft_probs, tree_tokens + (size_t)b * (size_t)N,
                tree_parents + (size_t)b * (size_t)N, num_nodes[b], temperature[b], b, N, V, ua,
                ue, out_ids + (size_t)b * (size_t)N, &out_num_accepted[b], &out_last_node[b],
                node_diag ? node_diag + (size_t)b * (size_t)N * ORACLE_ROW_W : NULL,
                req_diag ? req_diag + (size_t)b * ORACLE_REQ_W : NULL, probe ? probe[b] : -1, l,
                r, w);
            if (rc != 0) ++bad;
        }
        free(scratch);
    }
    return bad;
}

/* Philox blocks for a list of counters, for cross-checking other copies of
 * the generator: out[4*i..4*i+3] = Philox(key, ctr[4*i..4*i+3]). */
void oracle_philox_blocks(const uint32_t* ctrs, const uint32_t key[2], int64_t n, uint32_t* out) {
    for (int64_t i = 0; i < n; ++i) oracle_philox4x32_10(ctrs + 4 * i, key, out + 4 * i);
}
