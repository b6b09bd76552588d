/*
 * lla_oracle.c -- plain, slow fp64 CPU oracle for log-linear attention in its
 * Log-Linear Mamba-2 form.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  The CUDA library never
 * includes, links or calls anything in this directory, and this file includes
 * nothing from the CUDA library.
 *
 * Sources (page titles, sections):
 *   "Log-Linear Attention" (gist.science 2506.04761), technical summary
 *     §2.2 "数学的定式化": the output is a lambda-weighted sum over levels of
 *     q_t^T S_t^(l), with the prefix [0,t) split into at most L disjoint
 *     Fenwick-tree buckets, one hidden state per bucket.
 *   same page, §2.3 "効率的なアルゴリズム": the decode form is recurrent and
 *     touches O(log T) states per step.
 *   same page, §3: the Mamba-2 instance ("Log-Linear Mamba-2"): a scalar
 *     per-head gate g_t <= 0, G = cumsum(g), decay exp(G_t - G_s).
 *
 * Conventions (readings where the pages are silent):
 *   - positions are 0-based; the buckets of query t partition [0, t);
 *   - level of a key s for query t is bit_length(t XOR s): 0 for s == t, and
 *     for s < t the level l >= 1 bucket has 2^(l-1) members;
 *   - G_t = sum_{r<=t} g_r (inclusive), so the diagonal term has decay 1;
 *   - L = 1 + bit_length(T-1) weights per token; lambda is [B,H,T,L].
 *
 * Every array is C-contiguous fp64.  Layouts:
 *   q [B,H,T,dk], k [B,H,T,dk], v [B,H,T,dv], g [B,H,T], lam [B,H,T,L],
 *   out [B,H,T,dv].
 * Functions return 0 on success and a negative number on a bad argument.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Number of binary digits of x (0 for x == 0), by repeated halving. */
static int bit_length(uint64_t x)
{
    int n = 0;
    while (x) {
        n++;
        x >>= 1;
    }
    return n;
}

/* Number of trailing zero bits of x > 0, by repeated halving. */
static int trailing_zeros(uint64_t x)
{
    int n = 0;
    while ((x & 1u) == 0u) {
        n++;
        x >>= 1;
    }
    return n;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

int oracle_level(int64_t t, int64_t s)
{
    return bit_length((uint64_t)(t ^ s));
}

/* Inclusive running sum of one head's gates: G_t = g_0 + ... + g_t. */
static void cumsum(const double *g, int64_t T, double *G)
{
    double acc = 0.0;
    for (int64_t t = 0; t < T; t++) {
        acc += g[t];
        G[t] = acc;
    }
}

static double dot(const double *a, const double *b, int64_t n)
{
    double acc = 0.0;
    for (int64_t i = 0; i < n; i++)
        acc += a[i] * b[i];
    return acc;
}

/*
 * The defining double sum ("Log-Linear Attention" §2.2 with the Mamba-2 gate
 * of §3), written out term by term:
 *     o_t = sum_{s<=t} lam_t[level(t,s)] * exp(G_t - G_s) * (q_t . k_s) * v_s
 * O(T^2 (dk+dv)) per (batch, head).
 */
int oracle_naive(const double *q, const double *k, const double *v,
                 const double *g, const double *lam, double *out,
                 int64_t B, int64_t H, int64_t T, int64_t dk, int64_t dv,
                 int64_t L)
{
    if (B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0 || L <= 0)
        return -1;
    if (T > 0 && bit_length((uint64_t)(T - 1)) > L - 1)
        return -2;
    int64_t BH = B * H;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t bh = 0; bh < BH; bh++) {
        const double *qh = q + bh * T * dk;
        const double *kh = k + bh * T * dk;
        const double *vh = v + bh * T * dv;
        const double *gh = g + bh * T;
        const double *lh = lam + bh * T * L;
        double *oh = out + bh * T * dv;
        double *G = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
        if (!G) {
            bad |= 1;
            continue;
        }
        cumsum(gh, T, G);
        for (int64_t t = 0; t < T; t++) {
            double *o = oh + t * dv;
            for (int64_t j = 0; j < dv; j++)
                o[j] = 0.0;
            for (int64_t s = 0; s <= t; s++) {
                int lev = oracle_level(t, s);
                double w = lh[t * L + lev] * exp(G[t] - G[s]) *
                           dot(qh + t * dk, kh + s * dk, dk);
                const double *vs = vh + s * dv;
                for (int64_t j = 0; j < dv; j++)
                    o[j] += w * vs[j];
            }
        }
        free(G);
    }
    return bad ? -3 : 0;
}

/*
 * The same double sum for selected rows only: one (batch, head) slice
 * q [T,dk], k [T,dk], v [T,dv], g [T], lam [T,L]; rows[n] lists token
 * indices t, out [n,dv] receives o_t.  O(n T (dk+dv)); lets a test check
 * single outputs of long sequences.
 */
int oracle_naive_rows(const double *q, const double *k, const double *v,
                      const double *g, const double *lam, const int64_t *rows,
                      double *out, int64_t n, int64_t T, int64_t dk, int64_t dv,
                      int64_t L)
{
    if (T < 0 || dk <= 0 || dv <= 0 || L <= 0 || n < 0)
        return -1;
    if (T > 0 && bit_length((uint64_t)(T - 1)) > L - 1)
        return -2;
    for (int64_t i = 0; i < n; i++)
        if (rows[i] < 0 || rows[i] >= T)
            return -5;
    double *G = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    if (!G)
        return -3;
    cumsum(g, T, G);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n; i++) {
        int64_t t = rows[i];
        double *o = out + i * dv;
        for (int64_t j = 0; j < dv; j++)
            o[j] = 0.0;
        for (int64_t s = 0; s <= t; s++) {
            int lev = oracle_level(t, s);
            double w = lam[t * L + lev] * exp(G[t] - G[s]) * dot(q + t * dk, k + s * dk, dk);
            for (int64_t j = 0; j < dv; j++)
                o[j] += w * v[s * dv + j];
        }
    }
    free(G);
    return 0;
}

/*
 * Per-token Fenwick recurrence ("Log-Linear Attention" §2.2 buckets, §2.3
 * recurrent decode), with the decay applied eagerly to every live state.
 *
 * Before token t, slot l (l >= 1) holds, when live, the state of one Fenwick
 * bucket of [0, t):  S_l = sum_{s in bucket} exp(G_{t-1} - G_s) k_s v_s^T.
 * Step t:
 *   1. decay every live slot by exp(g_t)   (now decayed to t);
 *   2. o_t = lam_t[0] (q_t.k_t) v_t + sum_{live l} lam_t[l] q_t^T S_l;
 *   3. Fenwick insert of token t, a binary-counter carry: the new bucket
 *      joins token t with the live slots 1..m, m = trailing zeros of t+1;
 *      slots 1..m are emptied and slot m+1 receives the merged state.
 * The slots' liveness is tracked with explicit flags, not derived from bits
 * of t, so that the test suite can check it against the binary digits of t.
 * If live_count_out is non-NULL it receives, per (b,h,t), the number of live
 * slots read at step 2.
 */
int oracle_fenwick(const double *q, const double *k, const double *v,
                   const double *g, const double *lam, double *out,
                   int64_t B, int64_t H, int64_t T, int64_t dk, int64_t dv,
                   int64_t L, int32_t *live_count_out)
{
    if (B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0 || L <= 0)
        return -1;
    if (T > 0 && bit_length((uint64_t)(T - 1)) > L - 1)
        return -2;
    /* slots 1..L: the carry after the last token may reach level
       bit_length(T) = L when T is a power of two. */
    const int64_t nslot = L + 1;
    int64_t BH = B * H;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t bh = 0; bh < BH; bh++) {
        const double *qh = q + bh * T * dk;
        const double *kh = k + bh * T * dk;
        const double *vh = v + bh * T * dv;
        const double *gh = g + bh * T;
        const double *lh = lam + bh * T * L;
        double *oh = out + bh * T * dv;
        double *S = (double *)calloc((size_t)(nslot * dk * dv), sizeof(double));
        double *merged = (double *)malloc(sizeof(double) * (size_t)(dk * dv));
        int *live = (int *)calloc((size_t)nslot, sizeof(int));
        if (!S || !merged || !live) {
            free(S);
            free(merged);
            free(live);
            bad |= 1;
            continue;
        }
        for (int64_t t = 0; t < T; t++) {
            const double *qt = qh + t * dk;
            const double *kt = kh + t * dk;
            const double *vt = vh + t * dv;
            const double *lt = lh + t * L;
            double *o = oh + t * dv;
            double decay = exp(gh[t]);
            /* 1. decay */
            for (int64_t l = 1; l < nslot; l++) {
                if (!live[l])
                    continue;
                double *Sl = S + l * dk * dv;
                for (int64_t e = 0; e < dk * dv; e++)
                    Sl[e] *= decay;
            }
            /* 2. read-out */
            double diag = lt[0] * dot(qt, kt, dk);
            for (int64_t j = 0; j < dv; j++)
                o[j] = diag * vt[j];
            int nlive = 0;
            for (int64_t l = 1; l < nslot; l++) {
                if (!live[l])
                    continue;
                nlive++;
                if (l >= L) {
                    bad |= 2; /* a live bucket without a lambda entry */
                    continue;
                }
                const double *Sl = S + l * dk * dv;
                for (int64_t j = 0; j < dv; j++) {
                    double acc = 0.0;
                    for (int64_t i = 0; i < dk; i++)
                        acc += qt[i] * Sl[i * dv + j];
                    o[j] += lt[l] * acc;
                }
            }
            if (live_count_out)
                live_count_out[bh * T + t] = nlive;
            /* 3. insert token t */
            int m = trailing_zeros((uint64_t)(t + 1));
            if (m + 1 >= nslot) {
                bad |= 4;
                continue;
            }
            for (int64_t i = 0; i < dk; i++)
                for (int64_t j = 0; j < dv; j++)
                    merged[i * dv + j] = kt[i] * vt[j];
            for (int64_t l = 1; l <= m; l++) {
                if (!live[l]) {
                    bad |= 8; /* a carry through an empty slot */
                    continue;
                }
                const double *Sl = S + l * dk * dv;
                for (int64_t e = 0; e < dk * dv; e++)
                    merged[e] += Sl[e];
                live[l] = 0;
            }
            if (live[m + 1])
                bad |= 16; /* the carry target must be empty */
            memcpy(S + (m + 1) * dk * dv, merged, sizeof(double) * (size_t)(dk * dv));
            live[m + 1] = 1;
        }
        free(S);
        free(merged);
        free(live);
    }
    return bad ? -(8 + bad) : 0;
}

/*
 * One decode step on a lazily decayed level state (the recurrent form of
 * "Log-Linear Attention" §2.3).  The state of one (batch, head):
 *   S [Ls, dk, dv]: slot i holds level i+1;
 *   d [Ls]:         log-decay; the level's true state is exp(d) * S.
 * Slot i is live for token index t iff bit i of t is set.  The step:
 *   1. d_l += g for every live slot;
 *   2. o = lam[0] (q.k) v + sum_{live l} lam[l] exp(d_l) q^T S_l;
 *   3. m = trailing zeros of t+1:
 *        S_{m+1} = k v^T + sum_{l=1..m} exp(d_l) S_l,  d_{m+1} = 0.
 * Arguments for one batch of independent (batch, head) pairs, C-contiguous:
 *   S [B,H,Ls,dk,dv], d [B,H,Ls], q,k [B,H,dk], v [B,H,dv], g [B,H],
 *   lam [B,H,Ls+1], out [B,H,dv], pos [B] (token index t of the step).
 * Returns -4 if some t has bit_length(t+1) > Ls (the state has no room).
 */
int oracle_decode_step(double *S, double *d, const double *q, const double *k,
                       const double *v, const double *g, const double *lam,
                       double *out, const int64_t *pos, int64_t B, int64_t H,
                       int64_t dk, int64_t dv, int64_t Ls)
{
    if (B < 0 || H < 0 || dk <= 0 || dv <= 0 || Ls <= 0)
        return -1;
    for (int64_t b = 0; b < B; b++)
        if (pos[b] < 0 || bit_length((uint64_t)(pos[b] + 1)) > Ls)
            return -4;
    int64_t BH = B * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < BH; bh++) {
        int64_t t = pos[bh / H];
        double *Sh = S + bh * Ls * dk * dv;
        double *dh = d + bh * Ls;
        const double *qh = q + bh * dk;
        const double *kh = k + bh * dk;
        const double *vh = v + bh * dv;
        const double *lh = lam + bh * (Ls + 1);
        double *o = out + bh * dv;
        for (int64_t i = 0; i < Ls; i++)
            if ((t >> i) & 1)
                dh[i] += g[bh];
        double diag = lh[0] * dot(qh, kh, dk);
        for (int64_t j = 0; j < dv; j++)
            o[j] = diag * vh[j];
        for (int64_t i = 0; i < Ls; i++) {
            if (!((t >> i) & 1))
                continue;
            double w = lh[i + 1] * exp(dh[i]);
            const double *Si = Sh + i * dk * dv;
            for (int64_t j = 0; j < dv; j++) {
                double acc = 0.0;
                for (int64_t r = 0; r < dk; r++)
                    acc += qh[r] * Si[r * dv + j];
                o[j] += w * acc;
            }
        }
        int m = trailing_zeros((uint64_t)(t + 1));
        double *Snew = Sh + (int64_t)m * dk * dv;
        /* the target slot m is dead for t (bit m of t is 0), so it can be
           overwritten only after the sources 0..m-1 are folded in */
        double *acc = (double *)malloc(sizeof(double) * (size_t)(dk * dv));
        for (int64_t r = 0; r < dk; r++)
            for (int64_t j = 0; j < dv; j++)
                acc[r * dv + j] = kh[r] * vh[j];
        for (int64_t i = 0; i < m; i++) {
            double w = exp(dh[i]);
            const double *Si = Sh + i * dk * dv;
            for (int64_t e = 0; e < dk * dv; e++)
                acc[e] += w * Si[e];
        }
        memcpy(Snew, acc, sizeof(double) * (size_t)(dk * dv));
        dh[m] = 0.0;
        free(acc);
    }
    return 0;
}

/*
 * The decode state of one prefix, straight from the definition: for query
 * index pos, every key s < pos goes to level l = bit_length(pos XOR s) >= 1,
 * decayed to the last prefix token pos-1:
 *     S_l = sum_{s<pos, level(pos,s)=l} exp(G_{pos-1} - G_s) k_s v_s^T,
 * stored in slot l-1 with log-decay 0.  Slots with no member are zero.
 * Arguments: k [B,H,Tp,dk], v [B,H,Tp,dv], g [B,H,Tp] hold prefixes of
 * length Tp >= max(pos); pos [B]; S out [B,H,Ls,dk,dv]; d out [B,H,Ls].
 */
int oracle_state_closed_form(const double *k, const double *v, const double *g,
                             const int64_t *pos, double *S, double *d,
                             int64_t B, int64_t H, int64_t Tp, int64_t dk,
                             int64_t dv, int64_t Ls)
{
    if (B < 0 || H < 0 || Tp < 0 || dk <= 0 || dv <= 0 || Ls <= 0)
        return -1;
    for (int64_t b = 0; b < B; b++)
        if (pos[b] < 0 || pos[b] > Tp || bit_length((uint64_t)pos[b]) > Ls)
            return -4;
    int64_t BH = B * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < BH; bh++) {
        int64_t p = pos[bh / H];
        const double *kh = k + bh * Tp * dk;
        const double *vh = v + bh * Tp * dv;
        const double *gh = g + bh * Tp;
        double *Sh = S + bh * Ls * dk * dv;
        double *dh = d + bh * Ls;
        memset(Sh, 0, sizeof(double) * (size_t)(Ls * dk * dv));
        for (int64_t i = 0; i < Ls; i++)
            dh[i] = 0.0;
        /* G_{p-1} - G_s = g_{s+1} + ... + g_{p-1}, accumulated backwards */
        double tail = 0.0;
        for (int64_t s = p - 1; s >= 0; s--) {
            int lev = oracle_level(p, s);
            double w = exp(tail);
            double *Sl = Sh + (int64_t)(lev - 1) * dk * dv;
            const double *ks = kh + s * dk;
            const double *vs = vh + s * dv;
            for (int64_t r = 0; r < dk; r++)
                for (int64_t j = 0; j < dv; j++)
                    Sl[r * dv + j] += w * ks[r] * vs[j];
            tail += gh[s];
        }
    }
    return 0;
}

/*
 * Plain gated linear attention (the Mamba-2 scalar-gate scan the pages build
 * on): one state, S_t = exp(g_t) S_{t-1} + k_t v_t^T, o_t = S_t^T q_t.
 * Log-linear attention with every lambda equal to 1 reduces to this.
 */
int oracle_ssd(const double *q, const double *k, const double *v,
               const double *g, double *out, int64_t B, int64_t H, int64_t T,
               int64_t dk, int64_t dv)
{
    if (B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0)
        return -1;
    int64_t BH = B * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < BH; bh++) {
        const double *qh = q + bh * T * dk;
        const double *kh = k + bh * T * dk;
        const double *vh = v + bh * T * dv;
        const double *gh = g + bh * T;
        double *oh = out + bh * T * dv;
        double *S = (double *)calloc((size_t)(dk * dv), sizeof(double));
        for (int64_t t = 0; t < T; t++) {
            double a = exp(gh[t]);
            for (int64_t r = 0; r < dk; r++)
                for (int64_t j = 0; j < dv; j++)
                    S[r * dv + j] = a * S[r * dv + j] + kh[t * dk + r] * vh[t * dv + j];
            for (int64_t j = 0; j < dv; j++) {
                double acc = 0.0;
                for (int64_t r = 0; r < dk; r++)
                    acc += qh[t * dk + r] * S[r * dv + j];
                oh[t * dv + j] = acc;
            }
        }
        free(S);
    }
    return 0;
}

/*
 * Per-(token, head) level weights from a two-layer MLP ("Adaptive memory
 * decay for Log-Linear Attention", §Method "LambdaMLPSoftplus"):
 *     h = d W1,   lambda = softplus(h W2 + b),
 * hidden width 2L, no activation between the layers.  Reading: d is one
 * vector of width Dd per (token, head) and the weights are shared by heads.
 * d [N,Dd], W1 [Dd,2L], W2 [2L,L], b [L] -> out [N,L]; softplus(z) =
 * log(1 + exp(z)), evaluated as max(z,0) + log1p(exp(-|z|)).
 */
int oracle_lambda_mlp(const double *d, const double *W1, const double *W2,
                      const double *b, double *out, int64_t N, int64_t Dd,
                      int64_t L)
{
    if (N < 0 || Dd <= 0 || L <= 0)
        return -1;
    const int64_t Hd = 2 * L;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; n++) {
        double h[2 * 64];
        if (Hd > 2 * 64)
            continue;
        for (int64_t j = 0; j < Hd; j++) {
            double acc = 0.0;
            for (int64_t k = 0; k < Dd; k++)
                acc += d[n * Dd + k] * W1[k * Hd + j];
            h[j] = acc;
        }
        for (int64_t l = 0; l < L; l++) {
            double z = b[l];
            for (int64_t j = 0; j < Hd; j++)
                z += h[j] * W2[j * L + l];
            out[n * L + l] = (z > 0.0 ? z : 0.0) + log1p(exp(-fabs(z)));
        }
    }
    return L > 64 ? -2 : 0;
}

/*
 * Gradients of L = sum_t dout_t . o_t with o_t the defining double sum of
 * "Log-Linear Attention" §2.2 (Mamba-2 gate of §3).  The pages print no
 * backward; each term below is the derivative of one summand
 *     a_ts = lam_t[l] * E_ts * (q_t . k_s) * (dout_t . v_s),
 *     E_ts = exp(G_t - G_s),  l = level(t,s),  s <= t,
 * accumulated pair by pair:
 *     dq_t      += lam_t[l] E_ts (dout_t . v_s) k_s
 *     dk_s      += lam_t[l] E_ts (dout_t . v_s) q_t
 *     dv_s      += lam_t[l] E_ts (q_t . k_s) dout_t
 *     dlam_t[l] += E_ts (q_t . k_s)(dout_t . v_s)
 *     dG_t += a_ts,  dG_s -= a_ts
 * and, since G_u = g_0 + ... + g_u, dg_r = sum_{u >= r} dG_u.
 * Arrays as for oracle_naive; dout [B,H,T,dv]; outputs dq [B,H,T,dk],
 * dk [B,H,T,dk], dv [B,H,T,dv], dg [B,H,T], dlam [B,H,T,L] (overwritten).
 */
int oracle_backward(const double *q, const double *k, const double *v,
                    const double *g, const double *lam, const double *dout,
                    double *dq, double *dk, double *dv, double *dg,
                    double *dlam, int64_t B, int64_t H, int64_t T, int64_t Dk,
                    int64_t Dv, int64_t L)
{
    if (B < 0 || H < 0 || T < 0 || Dk <= 0 || Dv <= 0 || L <= 0)
        return -1;
    if (T > 0 && bit_length((uint64_t)(T - 1)) > L - 1)
        return -2;
    int64_t BH = B * H;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t bh = 0; bh < BH; bh++) {
        const double *qh = q + bh * T * Dk, *kh = k + bh * T * Dk;
        const double *vh = v + bh * T * Dv, *dh = dout + bh * T * Dv;
        const double *lh = lam + bh * T * L;
        double *dqh = dq + bh * T * Dk, *dkh = dk + bh * T * Dk;
        double *dvh = dv + bh * T * Dv, *dgh = dg + bh * T;
        double *dlh = dlam + bh * T * L;
        memset(dqh, 0, sizeof(double) * (size_t)(T * Dk));
        memset(dkh, 0, sizeof(double) * (size_t)(T * Dk));
        memset(dvh, 0, sizeof(double) * (size_t)(T * Dv));
        memset(dlh, 0, sizeof(double) * (size_t)(T * L));
        double *G = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
        double *dG = (double *)calloc((size_t)(T > 0 ? T : 1), sizeof(double));
        if (!G || !dG) {
            free(G);
            free(dG);
            bad |= 1;
            continue;
        }
        cumsum(g + bh * T, T, G);
        for (int64_t t = 0; t < T; t++) {
            for (int64_t s = 0; s <= t; s++) {
                int lev = oracle_level(t, s);
                double E = exp(G[t] - G[s]);
                double qk = dot(qh + t * Dk, kh + s * Dk, Dk);
                double ov = dot(dh + t * Dv, vh + s * Dv, Dv);
                double A = lh[t * L + lev] * E;
                for (int64_t r = 0; r < Dk; r++) {
                    dqh[t * Dk + r] += A * ov * kh[s * Dk + r];
                    dkh[s * Dk + r] += A * ov * qh[t * Dk + r];
                }
                for (int64_t c = 0; c < Dv; c++)
                    dvh[s * Dv + c] += A * qk * dh[t * Dv + c];
                dlh[t * L + lev] += E * qk * ov;
                dG[t] += A * qk * ov;
                dG[s] -= A * qk * ov;
            }
        }
        double run = 0.0;
        for (int64_t r = T - 1; r >= 0; r--) {
            run += dG[r];
            dgh[r] = run;
        }
        free(G);
        free(dG);
    }
    return bad ? -3 : 0;
}

/*
 * Log-Linear Gated DeltaNet.  "Log-Linear Attention" §3 names the variant
 * and says it keeps the base model's structure and adds the hierarchical
 * (Fenwick) mask; it prints no formula.  Reading taken: every Fenwick
 * bucket keeps its own state, all states follow the Gated DeltaNet
 * transition of each new token, and the read-out weights them by lambda:
 *     A_r = alpha_r (I - beta_r k_r k_r^T),  alpha_r = exp(g_r),
 *     o_t = sum_{s<=t} lam_t[level(t,s)] beta_s v_s (k_s^T A_{s+1} ... A_t q_t).
 * With lambda = 1 this is Gated DeltaNet (sum of the bucket states = its
 * single state); with mutually orthogonal keys the transitions reduce to
 * the scalar decay and it is Log-Linear Mamba-2 with values beta_s v_s.
 * Arrays as for oracle_naive plus beta [B,H,T].
 */

/* x <- A_r x for one token r. */
static void gdn_apply(double *x, const double *kr, double alpha, double beta,
                      int64_t dk)
{
    double c = beta * dot(kr, x, dk);
    for (int64_t i = 0; i < dk; i++)
        x[i] = alpha * (x[i] - c * kr[i]);
}

/* Pair form: for each query t walk s = t, t-1, ..., 0 carrying
   x = A_{s+1} ... A_t q_t.  O(T^2 (dk+dv)) per (batch, head). */
int oracle_gdn_naive(const double *q, const double *k, const double *v,
                     const double *g, const double *beta, const double *lam,
                     double *out, int64_t B, int64_t H, int64_t T, int64_t dk,
                     int64_t dv, int64_t L)
{
    if (B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0 || L <= 0)
        return -1;
    if (T > 0 && bit_length((uint64_t)(T - 1)) > L - 1)
        return -2;
    int64_t BH = B * H;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t bh = 0; bh < BH; bh++) {
        const double *qh = q + bh * T * dk, *kh = k + bh * T * dk;
        const double *vh = v + bh * T * dv, *gh = g + bh * T, *bt = beta + bh * T;
        const double *lh = lam + bh * T * L;
        double *oh = out + bh * T * dv;
        double *x = (double *)malloc(sizeof(double) * (size_t)dk);
        if (!x) {
            bad |= 1;
            continue;
        }
        for (int64_t t = 0; t < T; t++) {
            double *o = oh + t * dv;
            for (int64_t j = 0; j < dv; j++)
                o[j] = 0.0;
            memcpy(x, qh + t * dk, sizeof(double) * (size_t)dk);
            for (int64_t s = t; s >= 0; s--) {
                double w = lh[t * L + oracle_level(t, s)] * bt[s] * dot(kh + s * dk, x, dk);
                for (int64_t j = 0; j < dv; j++)
                    o[j] += w * vh[s * dv + j];
                gdn_apply(x, kh + s * dk, exp(gh[s]), bt[s], dk);
            }
        }
        free(x);
    }
    return bad ? -3 : 0;
}

/* S <- A S for a state S [dk][dv] (S = sum k v^T form), column by column. */
static void gdn_transition(double *S, const double *kt, double alpha,
                           double beta, int64_t dk, int64_t dv)
{
    for (int64_t j = 0; j < dv; j++) {
        double c = 0.0;
        for (int64_t i = 0; i < dk; i++)
            c += kt[i] * S[i * dv + j];
        c *= beta;
        for (int64_t i = 0; i < dk; i++)
            S[i * dv + j] = alpha * (S[i * dv + j] - c * kt[i]);
    }
}

/*
 * Recurrent form, per token t (states as in oracle_fenwick, S = sum k v^T):
 *   1. every live level state: S_l <- A_t S_l;
 *   2. o_t = lam_t[0] beta_t (q_t.k_t) v_t + sum_{live l} lam_t[l] S_l^T q_t;
 *   3. Fenwick insert: S_{m+1} = beta_t k_t v_t^T + sum_{l=1..m} S_l,
 *      m = trailing zeros of t+1.
 */
int oracle_gdn_fenwick(const double *q, const double *k, const double *v,
                       const double *g, const double *beta, const double *lam,
                       double *out, int64_t B, int64_t H, int64_t T, int64_t dk,
                       int64_t dv, int64_t L)
{
    if (B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0 || L <= 0)
        return -1;
    if (T > 0 && bit_length((uint64_t)(T - 1)) > L - 1)
        return -2;
    const int64_t nslot = L + 1;
    int64_t BH = B * H;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t bh = 0; bh < BH; bh++) {
        const double *qh = q + bh * T * dk, *kh = k + bh * T * dk;
        const double *vh = v + bh * T * dv, *gh = g + bh * T, *bt = beta + bh * T;
        const double *lh = lam + bh * T * L;
        double *oh = out + bh * T * dv;
        double *S = (double *)calloc((size_t)(nslot * dk * dv), sizeof(double));
        int *live = (int *)calloc((size_t)nslot, sizeof(int));
        if (!S || !live) {
            free(S);
            free(live);
            bad |= 1;
            continue;
        }
        for (int64_t t = 0; t < T; t++) {
            const double *qt = qh + t * dk, *kt = kh + t * dk, *vt = vh + t * dv;
            const double *lt = lh + t * L;
            double *o = oh + t * dv;
            for (int64_t l = 1; l < nslot; l++)
                if (live[l])
                    gdn_transition(S + l * dk * dv, kt, exp(gh[t]), bt[t], dk, dv);
            double diag = lt[0] * bt[t] * dot(qt, kt, dk);
            for (int64_t j = 0; j < dv; j++)
                o[j] = diag * vt[j];
            for (int64_t l = 1; l < nslot; l++) {
                if (!live[l])
                    continue;
                if (l >= L) {
                    bad |= 2;
                    continue;
                }
                const double *Sl = S + l * dk * dv;
                for (int64_t j = 0; j < dv; j++) {
                    double acc = 0.0;
                    for (int64_t i = 0; i < dk; i++)
                        acc += qt[i] * Sl[i * dv + j];
                    o[j] += lt[l] * acc;
                }
            }
            int m = trailing_zeros((uint64_t)(t + 1));
            if (m + 1 >= nslot) {
                bad |= 4;
                continue;
            }
            double *dst = S + (m + 1) * dk * dv;
            for (int64_t i = 0; i < dk; i++)
                for (int64_t j = 0; j < dv; j++)
                    dst[i * dv + j] = bt[t] * kt[i] * vt[j];
            for (int64_t l = 1; l <= m; l++) {
                const double *Sl = S + l * dk * dv;
                for (int64_t e = 0; e < dk * dv; e++)
                    dst[e] += Sl[e];
                live[l] = 0;
            }
            live[m + 1] = 1;
        }
        free(S);
        free(live);
    }
    return bad ? -(8 + bad) : 0;
}

/* The base model, Gated DeltaNet, with one state: S <- A_t S + beta_t k_t v_t^T,
   o_t = S^T q_t. */
int oracle_gdn_base(const double *q, const double *k, const double *v,
                    const double *g, const double *beta, double *out, int64_t B,
                    int64_t H, int64_t T, int64_t dk, int64_t dv)
{
    if (B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0)
        return -1;
    int64_t BH = B * H;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t bh = 0; bh < BH; bh++) {
        double *S = (double *)calloc((size_t)(dk * dv), sizeof(double));
        if (!S) {
            bad |= 1;
            continue;
        }
        for (int64_t t = 0; t < T; t++) {
            const double *qt = q + (bh * T + t) * dk, *kt = k + (bh * T + t) * dk;
            const double *vt = v + (bh * T + t) * dv;
            double bt = beta[bh * T + t];
            gdn_transition(S, kt, exp(g[bh * T + t]), bt, dk, dv);
            for (int64_t i = 0; i < dk; i++)
                for (int64_t j = 0; j < dv; j++)
                    S[i * dv + j] += bt * kt[i] * vt[j];
            double *o = out + (bh * T + t) * dv;
            for (int64_t j = 0; j < dv; j++) {
                double acc = 0.0;
                for (int64_t i = 0; i < dk; i++)
                    acc += qt[i] * S[i * dv + j];
                o[j] = acc;
            }
        }
        free(S);
    }
    return bad ? -3 : 0;
}

/*
 * One decode step of the recurrent form on an eager level state
 * S [B,H,Ls,dk,dv] (slot i = level i+1; slot i is live for token t iff
 * bit i of t is set): steps 1-3 of oracle_gdn_fenwick for the token index
 * t = pos[b].  q,k [B,H,dk], v [B,H,dv], g, beta [B,H], lam [B,H,Ls+1],
 * out [B,H,dv].  Returns -4 if some t has bit_length(t+1) > Ls.
 */
int oracle_gdn_decode_step(double *S, const double *q, const double *k,
                           const double *v, const double *g, const double *beta,
                           const double *lam, double *out, const int64_t *pos,
                           int64_t B, int64_t H, int64_t dk, int64_t dv, int64_t Ls)
{
    if (B < 0 || H < 0 || dk <= 0 || dv <= 0 || Ls <= 0)
        return -1;
    for (int64_t b = 0; b < B; b++)
        if (pos[b] < 0 || bit_length((uint64_t)(pos[b] + 1)) > Ls)
            return -4;
    for (int64_t bh = 0; bh < B * H; bh++) {
        const int64_t t = pos[bh / H];
        double *Sb = S + bh * Ls * dk * dv;
        const double *qt = q + bh * dk, *kt = k + bh * dk, *vt = v + bh * dv;
        const double *lt = lam + bh * (Ls + 1);
        const double bt = beta[bh];
        double *o = out + bh * dv;
        for (int64_t i = 0; i < Ls; i++)
            if ((t >> i) & 1)
                gdn_transition(Sb + i * dk * dv, kt, exp(g[bh]), bt, dk, dv);
        double diag = lt[0] * bt * dot(qt, kt, dk);
        for (int64_t j = 0; j < dv; j++)
            o[j] = diag * vt[j];
        for (int64_t i = 0; i < Ls; i++) {
            if (!((t >> i) & 1))
                continue;
            const double *Sl = Sb + i * dk * dv;
            for (int64_t j = 0; j < dv; j++) {
                double acc = 0.0;
                for (int64_t r = 0; r < dk; r++)
                    acc += qt[r] * Sl[r * dv + j];
                o[j] += lt[i + 1] * acc;
            }
        }
        int m = trailing_zeros((uint64_t)(t + 1));
        double *dst = Sb + m * dk * dv;
        double *tmp = (double *)malloc(sizeof(double) * (size_t)(dk * dv));
        if (!tmp)
            return -3;
        for (int64_t r = 0; r < dk; r++)
            for (int64_t j = 0; j < dv; j++)
                tmp[r * dv + j] = bt * kt[r] * vt[j];
        for (int64_t i = 0; i < m; i++)
            for (int64_t e = 0; e < dk * dv; e++)
                tmp[e] += Sb[i * dk * dv + e];
        memcpy(dst, tmp, sizeof(double) * (size_t)(dk * dv));
        free(tmp);
    }
    return 0;
}

/*
 * The backward of oracle_backward at selected rows only, for one (batch,
 * head) slice q,k [T,dk], v,dout [T,dv], g [T], lam [T,L]:
 *   query rows tq[nq]: dq [nq,dk], dlam [nq,L]  (sums over s <= t)
 *   key rows   ts[ns]: dk [ns,dk], dv [ns,dv]   (sums over t >= s)
 * O((nq + ns) T (dk+dv)); lets a test check single rows of long sequences.
 */
int oracle_backward_rows(const double *q, const double *k, const double *v,
                         const double *g, const double *lam, const double *dout,
                         const int64_t *tq, int64_t nq, const int64_t *ts, int64_t ns,
                         double *dq, double *dlam, double *dk, double *dv,
                         int64_t T, int64_t Dk, int64_t Dv, int64_t L)
{
    if (T < 0 || Dk <= 0 || Dv <= 0 || L <= 0 || nq < 0 || ns < 0)
        return -1;
    if (T > 0 && bit_length((uint64_t)(T - 1)) > L - 1)
        return -2;
    for (int64_t i = 0; i < nq; i++)
        if (tq[i] < 0 || tq[i] >= T)
            return -5;
    for (int64_t i = 0; i < ns; i++)
        if (ts[i] < 0 || ts[i] >= T)
            return -5;
    double *G = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    if (!G)
        return -3;
    cumsum(g, T, G);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nq; i++) {
        const int64_t t = tq[i];
        double *dqi = dq + i * Dk, *dli = dlam + i * L;
        memset(dqi, 0, sizeof(double) * (size_t)Dk);
        memset(dli, 0, sizeof(double) * (size_t)L);
        for (int64_t s = 0; s <= t; s++) {
            int lev = oracle_level(t, s);
            double E = exp(G[t] - G[s]);
            double qk = dot(q + t * Dk, k + s * Dk, Dk);
            double ov = dot(dout + t * Dv, v + s * Dv, Dv);
            double A = lam[t * L + lev] * E;
            for (int64_t r = 0; r < Dk; r++)
                dqi[r] += A * ov * k[s * Dk + r];
            dli[lev] += E * qk * ov;
        }
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < ns; i++) {
        const int64_t s = ts[i];
        double *dki = dk + i * Dk, *dvi = dv + i * Dv;
        memset(dki, 0, sizeof(double) * (size_t)Dk);
        memset(dvi, 0, sizeof(double) * (size_t)Dv);
        for (int64_t t = s; t < T; t++) {
            int lev = oracle_level(t, s);
            double A = lam[t * L + lev] * exp(G[t] - G[s]);
            double qk = dot(q + t * Dk, k + s * Dk, Dk);
            double ov = dot(dout + t * Dv, v + s * Dv, Dv);
            for (int64_t r = 0; r < Dk; r++)
                dki[r] += A * ov * q[t * Dk + r];
            for (int64_t c = 0; c < Dv; c++)
                dvi[c] += A * qk * dout[t * Dv + c];
        }
    }
    free(G);
    return 0;
}
