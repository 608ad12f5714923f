/*
 * linattn_oracle.c -- plain FP64 CPU oracle for normalised causal linear
 * attention with a recurrent S/z state.  TEST INFRASTRUCTURE ONLY: nothing in
 * the product path links, loads or calls this file; only the test-suite, the
 * smoke check and the benchmark's CPU-baseline leg do.
 *
 * Sources (web pages; cited by title and section):
 *   [LA]  "Linear attention：把历史写进状态" (hs-black.github.io, posts/linear-attention)
 *   [LC]  "45. Linear Attention and Recurrent State | 线性注意力与递推状态"
 *         (datawhalechina llm-algo-leetcode, chapter 45)
 *   [LE]  "线性注意力架构演进：从 Transformer 瓶颈到高效推理" (ai-master.cc)
 *
 * Three independent routes to the same function, all in double precision:
 *   or_scan       the token recurrence (definition of the method)
 *                 [LA] "公式里的每个维度" (S_t, z_t, y_t), "每来一个 token，更新两个累加器"
 *                 (update before read), "加一个门：让旧记忆逐渐淡出" (scalar gate on S and z),
 *                 "ε 是数值保护" (y = num / (den + eps));
 *                 [LC] Step 2 and the reference answer of TODO 2/3.
 *   or_dense      the quadratic masked form A = (Q~K~^T) . M, Y = AV / rowsum(A)
 *                 [LA] "先确认我们在重排哪一种 attention"; gate weights are the product
 *                 of later gates, [LA] "遗忘门怎样改变历史的权重？" and Exercise 2.
 *   or_chunkwise  the chunk formula [LA] "一个 chunk 的输出由两部分组成"
 *                 (num = Q~c Sprev + [(Q~c K~c^T) . M] Vc, den likewise,
 *                 Snext = Sprev + K~c^T Vc, znext = zprev + sum of rows of K~c),
 *                 with the gate products inserted as that section asks for the gated
 *                 version (read: every term is multiplied by the product of the gates
 *                 that act on it between its write and its read; see or_chunkwise).
 *
 * A fourth routine, or_delta, is the delta-rule memory of [LA] "Delta rule：先读旧答案，
 * 再写误差" (a different update rule, without the normaliser; see its comment).
 *
 * Feature maps: ELU(x)+1 ([LA] "关键改写：让求和先发生"; [LE] feature_map), relu(x)+1
 * ([LC] reference answer of TODO 1) and the identity (so that the pages' worked
 * examples, which give feature values directly, can be replayed).
 *
 * Inputs are decoded exactly to double: FP64 as is, FP32 widened, BF16 widened
 * from its 16 stored bits (bits << 16 is the FP32 with the same value).
 * All arrays are row-major and contiguous:
 *   q, k [B,H,T,r]; v [B,H,T,dv]; alpha [B,H,T] (NULL: alpha == 1);
 *   S0 [B,H,r,dv], z0 [B,H,r] (NULL: zero); y [B,H,T,dv]; S [B,H,r,dv]; z [B,H,r].
 * Return value 0 on success, -1 on a bad argument.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { OR_F64 = 0, OR_F32 = 1, OR_BF16 = 2 };
enum { OR_PHI_ELU1 = 0, OR_PHI_RELU1 = 1, OR_PHI_IDENTITY = 2 };

static double decode(const void *base, int type, size_t idx)
{
    if (type == OR_F64) return ((const double *)base)[idx];
    if (type == OR_F32) return (double)((const float *)base)[idx];
    /* BF16: the upper 16 bits of an IEEE binary32. */
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ELU(x)+1 with the ELU parameter 1: x+1 for x>0, (e^x - 1) + 1 = e^x otherwise. */
static double phi(double x, int kind)
{
    if (kind == OR_PHI_ELU1) return x > 0.0 ? x + 1.0 : exp(x);
    if (kind == OR_PHI_RELU1) return (x > 0.0 ? x : 0.0) + 1.0;
    return x;
}

typedef struct {
    int B, H, T, r, dv, in_type, phi_kind, chunk;
    const void *q, *k, *v;
    const double *alpha, *S0, *z0;
    double eps;
    double *y, *S, *z;
} problem;

static int check(const problem *p)
{
    if (p->B < 1 || p->H < 1 || p->T < 1 || p->r < 1 || p->dv < 1) return -1;
    if (!p->q || !p->k || !p->v || !p->y || !p->S || !p->z) return -1;
    if (p->in_type < OR_F64 || p->in_type > OR_BF16) return -1;
    if (p->phi_kind < OR_PHI_ELU1 || p->phi_kind > OR_PHI_IDENTITY) return -1;
    return 0;
}

static double gate(const problem *p, size_t bh, int t)
{
    return p->alpha ? p->alpha[bh * (size_t)p->T + (size_t)t] : 1.0;
}

/* ------------------------------------------------------------------ scan -- */

/* One (b,h) sequence, token by token, state updated before it is read. */
static void scan_one(const problem *p, size_t bh, double *qt, double *kt, double *num)
{
    const int T = p->T, r = p->r, dv = p->dv;
    double *S = p->S + bh * (size_t)r * dv;
    double *z = p->z + bh * (size_t)r;
    if (p->S0) memcpy(S, p->S0 + bh * (size_t)r * dv, sizeof(double) * (size_t)r * dv);
    else memset(S, 0, sizeof(double) * (size_t)r * dv);
    if (p->z0) memcpy(z, p->z0 + bh * (size_t)r, sizeof(double) * (size_t)r);
    else memset(z, 0, sizeof(double) * (size_t)r);

    for (int t = 0; t < T; ++t) {
        const size_t row_qk = (bh * (size_t)T + (size_t)t) * (size_t)r;
        const size_t row_v = (bh * (size_t)T + (size_t)t) * (size_t)dv;
        const double a = gate(p, bh, t);
        for (int i = 0; i < r; ++i) {
            qt[i] = phi(decode(p->q, p->in_type, row_qk + i), p->phi_kind);
            kt[i] = phi(decode(p->k, p->in_type, row_qk + i), p->phi_kind);
        }
        /* S_t = a S_{t-1} + phi(k_t) v_t^T ;  z_t = a z_{t-1} + phi(k_t) */
        for (int i = 0; i < r; ++i) {
            double *Si = S + (size_t)i * dv;
            for (int j = 0; j < dv; ++j)
                Si[j] = a * Si[j] + kt[i] * decode(p->v, p->in_type, row_v + j);
            z[i] = a * z[i] + kt[i];
        }
        /* y_t = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps) */
        double den = 0.0;
        for (int j = 0; j < dv; ++j) num[j] = 0.0;
        for (int i = 0; i < r; ++i) {
            const double *Si = S + (size_t)i * dv;
            for (int j = 0; j < dv; ++j) num[j] += qt[i] * Si[j];
            den += qt[i] * z[i];
        }
        for (int j = 0; j < dv; ++j) p->y[row_v + j] = num[j] / (den + p->eps);
    }
}

typedef struct {
    const problem *p;
    size_t next;
    pthread_mutex_t lock;
} work_queue;

static void *scan_worker(void *arg)
{
    work_queue *w = (work_queue *)arg;
    const problem *p = w->p;
    double *buf = (double *)malloc(sizeof(double) * (2 * (size_t)p->r + (size_t)p->dv));
    if (!buf) return NULL;
    const size_t nbh = (size_t)p->B * (size_t)p->H;
    for (;;) {
        pthread_mutex_lock(&w->lock);
        size_t bh = w->next++;
        pthread_mutex_unlock(&w->lock);
        if (bh >= nbh) break;
        scan_one(p, bh, buf, buf + p->r, buf + 2 * (size_t)p->r);
    }
    free(buf);
    return NULL;
}

int or_num_cpus(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n < 1 ? 1 : (int)n;
}

int or_scan(int B, int H, int T, int r, int dv, const void *q, const void *k, const void *v,
            int in_type, const double *alpha, const double *S0, const double *z0, double eps,
            int phi_kind, int nthreads, double *y, double *S, double *z)
{
    problem p = {B, H, T, r, dv, in_type, phi_kind, 0, q, k, v, alpha, S0, z0, eps, y, S, z};
    if (check(&p)) return -1;
    const size_t nbh = (size_t)B * (size_t)H;
    if (nthreads <= 0) nthreads = or_num_cpus();
    if ((size_t)nthreads > nbh) nthreads = (int)nbh;
    work_queue w;
    w.p = &p;
    w.next = 0;
    pthread_mutex_init(&w.lock, NULL);
    if (nthreads == 1) {
        scan_worker(&w);
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        if (!th) return -1;
        for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, scan_worker, &w);
        for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&w.lock);
    return 0;
}

/* ----------------------------------------------------------------- dense -- */

/* Product of the gates alpha_{lo..hi} (inclusive); 1 for an empty range. */
static double gate_product(const problem *p, size_t bh, int lo, int hi)
{
    double g = 1.0;
    for (int u = lo; u <= hi; ++u) g *= gate(p, bh, u);
    return g;
}

/* Quadratic form on tiny inputs: every query row is an explicitly normalised
 * weighted average over the visible keys (the mask keeps past AND current),
 * weight_{t,s} = (q~_t . k~_s) * prod_{u=s+1..t} alpha_u, plus the carried-in
 * state S0/z0 weighted by prod_{u=0..t} alpha_u. */
int or_dense(int B, int H, int T, int r, int dv, const void *q, const void *k, const void *v,
             int in_type, const double *alpha, const double *S0, const double *z0, double eps,
             int phi_kind, double *y, double *S, double *z)
{
    problem p = {B, H, T, r, dv, in_type, phi_kind, 0, q, k, v, alpha, S0, z0, eps, y, S, z};
    if (check(&p)) return -1;
    double *Qf = (double *)malloc(sizeof(double) * (size_t)T * r);
    double *Kf = (double *)malloc(sizeof(double) * (size_t)T * r);
    double *A = (double *)malloc(sizeof(double) * (size_t)T * T);
    if (!Qf || !Kf || !A) { free(Qf); free(Kf); free(A); return -1; }
    for (size_t bh = 0; bh < (size_t)B * H; ++bh) {
        const size_t qk0 = bh * (size_t)T * r, v0 = bh * (size_t)T * dv;
        for (size_t e = 0; e < (size_t)T * r; ++e) {
            Qf[e] = phi(decode(q, in_type, qk0 + e), phi_kind);
            Kf[e] = phi(decode(k, in_type, qk0 + e), phi_kind);
        }
        /* A = (Q~ K~^T) . M, with M_{ts} = prod_{u=s+1..t} alpha_u for s <= t, else 0 */
        for (int t = 0; t < T; ++t)
            for (int s = 0; s < T; ++s) {
                double a = 0.0;
                if (s <= t) {
                    for (int i = 0; i < r; ++i) a += Qf[(size_t)t * r + i] * Kf[(size_t)s * r + i];
                    a *= gate_product(&p, bh, s + 1, t);
                }
                A[(size_t)t * T + s] = a;
            }
        const double *S0h = S0 ? S0 + bh * (size_t)r * dv : NULL;
        const double *z0h = z0 ? z0 + bh * (size_t)r : NULL;
        for (int t = 0; t < T; ++t) {
            const double carry = gate_product(&p, bh, 0, t);
            double rowsum = 0.0;
            for (int s = 0; s <= t; ++s) rowsum += A[(size_t)t * T + s];
            double den = rowsum;
            if (z0h)
                for (int i = 0; i < r; ++i) den += carry * Qf[(size_t)t * r + i] * z0h[i];
            for (int j = 0; j < dv; ++j) {
                double n = 0.0;
                for (int s = 0; s <= t; ++s)
                    n += A[(size_t)t * T + s] * decode(v, in_type, v0 + (size_t)s * dv + j);
                if (S0h)
                    for (int i = 0; i < r; ++i) n += carry * Qf[(size_t)t * r + i] * S0h[(size_t)i * dv + j];
                y[v0 + (size_t)t * dv + j] = n / (den + eps);
            }
        }
        /* Final state: every write decays by the gates that follow it. */
        double *Sh = S + bh * (size_t)r * dv, *zh = z + bh * (size_t)r;
        const double carry = gate_product(&p, bh, 0, T - 1);
        for (int i = 0; i < r; ++i) {
            zh[i] = z0h ? carry * z0h[i] : 0.0;
            for (int j = 0; j < dv; ++j) Sh[(size_t)i * dv + j] = S0h ? carry * S0h[(size_t)i * dv + j] : 0.0;
        }
        for (int s = 0; s < T; ++s) {
            const double w = gate_product(&p, bh, s + 1, T - 1);
            for (int i = 0; i < r; ++i) {
                zh[i] += w * Kf[(size_t)s * r + i];
                for (int j = 0; j < dv; ++j)
                    Sh[(size_t)i * dv + j] += w * Kf[(size_t)s * r + i] * decode(v, in_type, v0 + (size_t)s * dv + j);
            }
        }
    }
    free(Qf); free(Kf); free(A);
    return 0;
}

/* ------------------------------------------------------------- chunkwise -- */

/* Chunk formula.  For a chunk of n rows starting at token c0 (local indices 0..n-1):
 *   G_i    = prod_{u=0..i} alpha_{c0+u}          decay of the carried-in state at row i
 *   D_ij   = prod_{u=j+1..i} alpha_{c0+u}, j<=i  decay of row j's write when row i reads
 *   num_i  = G_i q~_i Sprev + sum_{j<=i} D_ij (q~_i . k~_j) v_j
 *   den_i  = G_i q~_i . zprev + sum_{j<=i} D_ij (q~_i . k~_j)
 *   y_i    = num_i / (den_i + eps)
 *   Snext  = G_{n-1} Sprev + sum_j D_{n-1,j} k~_j v_j^T,  znext likewise with k~_j.
 * With alpha == 1 every G and D is 1 and this is the page's ungated formula verbatim.
 * The last chunk may be shorter than C. */
int or_chunkwise(int B, int H, int T, int r, int dv, const void *q, const void *k, const void *v,
                 int in_type, const double *alpha, const double *S0, const double *z0,
                 double eps, int phi_kind, int C, double *y, double *S, double *z)
{
    problem p = {B, H, T, r, dv, in_type, phi_kind, C, q, k, v, alpha, S0, z0, eps, y, S, z};
    if (check(&p) || C < 1) return -1;
    double *Qc = (double *)malloc(sizeof(double) * (size_t)C * r);
    double *Kc = (double *)malloc(sizeof(double) * (size_t)C * r);
    double *Vc = (double *)malloc(sizeof(double) * (size_t)C * dv);
    double *P = (double *)malloc(sizeof(double) * (size_t)C * C);
    double *D = (double *)malloc(sizeof(double) * (size_t)C * C);
    double *G = (double *)malloc(sizeof(double) * (size_t)C);
    double *Sn = (double *)malloc(sizeof(double) * (size_t)r * dv);
    double *zn = (double *)malloc(sizeof(double) * (size_t)r);
    if (!Qc || !Kc || !Vc || !P || !D || !G || !Sn || !zn) {
        free(Qc); free(Kc); free(Vc); free(P); free(D); free(G); free(Sn); free(zn);
        return -1;
    }
    for (size_t bh = 0; bh < (size_t)B * H; ++bh) {
        double *Sh = S + bh * (size_t)r * dv, *zh = z + bh * (size_t)r;
        for (size_t e = 0; e < (size_t)r * dv; ++e) Sh[e] = S0 ? S0[bh * (size_t)r * dv + e] : 0.0;
        for (int i = 0; i < r; ++i) zh[i] = z0 ? z0[bh * (size_t)r + i] : 0.0;

        for (int c0 = 0; c0 < T; c0 += C) {
            const int n = (T - c0 < C) ? T - c0 : C;
            for (int t = 0; t < n; ++t)
                for (int i = 0; i < r; ++i) {
                    const size_t e = (bh * (size_t)T + (size_t)(c0 + t)) * r + i;
                    Qc[(size_t)t * r + i] = phi(decode(q, in_type, e), phi_kind);
                    Kc[(size_t)t * r + i] = phi(decode(k, in_type, e), phi_kind);
                }
            for (int t = 0; t < n; ++t)
                for (int j = 0; j < dv; ++j)
                    Vc[(size_t)t * dv + j] = decode(v, in_type, (bh * (size_t)T + (size_t)(c0 + t)) * dv + j);
            /* gate products inside the chunk */
            for (int i = 0; i < n; ++i) {
                G[i] = (i == 0 ? 1.0 : G[i - 1]) * gate(&p, bh, c0 + i);
                D[(size_t)i * C + i] = 1.0;
                for (int j = i - 1; j >= 0; --j)
                    D[(size_t)i * C + j] = D[(size_t)i * C + j + 1] * gate(&p, bh, c0 + j + 1);
            }
            /* P = Q~c K~c^T, kept only where the in-chunk causal mask allows (j <= i) */
            for (int i = 0; i < n; ++i)
                for (int j = 0; j <= i; ++j) {
                    double a = 0.0;
                    for (int f = 0; f < r; ++f) a += Qc[(size_t)i * r + f] * Kc[(size_t)j * r + f];
                    P[(size_t)i * C + j] = a * D[(size_t)i * C + j];
                }
            for (int i = 0; i < n; ++i) {
                /* inter-chunk read from the carried state, then the in-chunk part */
                double den = 0.0;
                for (int f = 0; f < r; ++f) den += Qc[(size_t)i * r + f] * zh[f];
                den *= G[i];
                for (int j = 0; j <= i; ++j) den += P[(size_t)i * C + j];
                for (int col = 0; col < dv; ++col) {
                    double inter = 0.0, intra = 0.0;
                    for (int f = 0; f < r; ++f) inter += Qc[(size_t)i * r + f] * Sh[(size_t)f * dv + col];
                    for (int j = 0; j <= i; ++j) intra += P[(size_t)i * C + j] * Vc[(size_t)j * dv + col];
                    y[(bh * (size_t)T + (size_t)(c0 + i)) * dv + col] = (G[i] * inter + intra) / (den + eps);
                }
            }
            /* state hand-off to the next chunk */
            const double Gl = G[n - 1];
            for (int f = 0; f < r; ++f) {
                double zacc = 0.0;
                for (int j = 0; j < n; ++j) zacc += D[(size_t)(n - 1) * C + j] * Kc[(size_t)j * r + f];
                zn[f] = Gl * zh[f] + zacc;
                for (int col = 0; col < dv; ++col) {
                    double sacc = 0.0;
                    for (int j = 0; j < n; ++j)
                        sacc += D[(size_t)(n - 1) * C + j] * Kc[(size_t)j * r + f] * Vc[(size_t)j * dv + col];
                    Sn[(size_t)f * dv + col] = Gl * Sh[(size_t)f * dv + col] + sacc;
                }
            }
            memcpy(Sh, Sn, sizeof(double) * (size_t)r * dv);
            memcpy(zh, zn, sizeof(double) * (size_t)r);
        }
    }
    free(Qc); free(Kc); free(Vc); free(P); free(D); free(G); free(Sn); free(zn);
    return 0;
}

/* ------------------------------------------------------------ delta rule -- */

/*
 * The delta rule ([LA] "Delta rule：先读旧答案，再写误差"): a fast-weight memory
 * without the normaliser.  For each token, first read the memory's current answer
 * for the key, then write back only the error, scaled by beta:
 *     p_t = S_{t-1}^T k_t,   e_t = v_t - p_t,   S_t = S_{t-1} + beta_t k_t e_t^T,
 * and the output reads the updated memory with the query, y_t = S_t^T q_t (read
 * after write, as for the accumulators).  q and k are used as given (the pages'
 * examples give them directly; [LA] "key 的范数决定了纠错力度" discusses their norm).
 *   q, k [B,H,T,r]; v [B,H,T,dv] (in_type); beta [B,H,T] (NULL: 1); S0 [B,H,r,dv]
 *   (NULL: zero); y [B,H,T,dv]; S [B,H,r,dv].
 */
typedef struct {
    int B, H, T, r, dv, in_type;
    const void *q, *k, *v;
    const double *beta, *S0;
    double *y, *S;
    size_t next;
    pthread_mutex_t lock;
} delta_problem;

static void delta_one(const delta_problem *p, size_t bh, double *kt, double *pe)
{
    const int T = p->T, r = p->r, dv = p->dv;
    double *S = p->S + bh * (size_t)r * dv;
    if (p->S0) memcpy(S, p->S0 + bh * (size_t)r * dv, sizeof(double) * (size_t)r * dv);
    else memset(S, 0, sizeof(double) * (size_t)r * dv);
    for (int t = 0; t < T; ++t) {
        const size_t row_qk = (bh * (size_t)T + (size_t)t) * (size_t)r;
        const size_t row_v = (bh * (size_t)T + (size_t)t) * (size_t)dv;
        const double beta = p->beta ? p->beta[bh * (size_t)T + (size_t)t] : 1.0;
        for (int i = 0; i < r; ++i) kt[i] = decode(p->k, p->in_type, row_qk + i);
        /* the memory's answer for k_t, then the error against v_t */
        for (int j = 0; j < dv; ++j) pe[j] = 0.0;
        for (int i = 0; i < r; ++i)
            for (int j = 0; j < dv; ++j) pe[j] += S[(size_t)i * dv + j] * kt[i];
        for (int j = 0; j < dv; ++j) pe[j] = decode(p->v, p->in_type, row_v + j) - pe[j];
        /* write back beta * k_t e_t^T */
        for (int i = 0; i < r; ++i)
            for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += beta * kt[i] * pe[j];
        /* y_t = S_t^T q_t */
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < r; ++i) acc += S[(size_t)i * dv + j] * decode(p->q, p->in_type, row_qk + i);
            p->y[row_v + j] = acc;
        }
    }
}

static void *delta_worker(void *arg)
{
    delta_problem *p = (delta_problem *)arg;
    double *buf = (double *)malloc(sizeof(double) * ((size_t)p->r + (size_t)p->dv));
    if (!buf) return NULL;
    const size_t nbh = (size_t)p->B * (size_t)p->H;
    for (;;) {
        pthread_mutex_lock(&p->lock);
        size_t bh = p->next++;
        pthread_mutex_unlock(&p->lock);
        if (bh >= nbh) break;
        delta_one(p, bh, buf, buf + p->r);
    }
    free(buf);
    return NULL;
}

int or_delta(int B, int H, int T, int r, int dv, const void *q, const void *k, const void *v, int in_type,
             const double *beta, const double *S0, int nthreads, double *y, double *S)
{
    if (B < 1 || H < 1 || T < 1 || r < 1 || dv < 1) return -1;
    if (!q || !k || !v || !y || !S) return -1;
    if (in_type < OR_F64 || in_type > OR_BF16) return -1;
    delta_problem p = {B, H, T, r, dv, in_type, q, k, v, beta, S0, y, S, 0, PTHREAD_MUTEX_INITIALIZER};
    const size_t nbh = (size_t)B * (size_t)H;
    if (nthreads <= 0) nthreads = or_num_cpus();
    if ((size_t)nthreads > nbh) nthreads = (int)nbh;
    if (nthreads == 1) {
        delta_worker(&p);
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        if (!th) return -1;
        for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, delta_worker, &p);
        for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    return 0;
}

/* -------------------------------------------------------------- backward -- */

/*
 * Gradients of the token recurrence (or_scan) for a loss L whose derivatives
 * with respect to the outputs are given: dy [B,H,T,dv], and optionally dS_T
 * [B,H,r,dv], dz_T [B,H,r] (NULL: zero).  The pages give no backward formula;
 * this is the chain rule applied to the recurrence of [LA] "公式里的每个维度"
 * and "加一个门：让旧记忆逐渐淡出", step by step in reverse:
 *   with y_t = n_t / d_t,  n_t = S_t^T q~_t,  d_t = q~_t . z_t + eps:
 *     dn_t = dy_t / d_t,   dd_t = -(dy_t . y_t) / d_t;
 *   G_t = dL/dS_t = q~_t dn_t^T + alpha_{t+1} G_{t+1}   (G_T from dS_T),
 *   g_t = dL/dz_t = dd_t q~_t  + alpha_{t+1} g_{t+1}    (g_T from dz_T);
 *     dq~_t = S_t dn_t + dd_t z_t,   dk~_t = G_t v_t + g_t,   dv_t = G_t^T k~_t,
 *     dalpha_t = <G_t, S_{t-1}> + <g_t, z_{t-1}>,   dS0 = alpha_1 G_1,  dz0 = alpha_1 g_1;
 *   dq_t = dq~_t * phi'(q_t), dk_t = dk~_t * phi'(k_t), phi'(x) = 1 for x > 0 and
 *   e^x otherwise (ELU+1), 0 otherwise for relu+1, 1 for the identity.
 * The reverse sweep needs S_t and S_{t-1} at every step.  They are recomputed
 * segment by segment from states saved every kSeg tokens during a first forward
 * sweep; the recomputation repeats the forward arithmetic exactly, so the states
 * are the same numbers as in or_scan.
 *   dq, dk [B,H,T,r]; dv [B,H,T,dv]; dalpha [B,H,T] (written when alpha is given);
 *   dS0 [B,H,r,dv]; dz0 [B,H,r].
 */
enum { kSeg = 64 };

typedef struct {
    problem f;                 /* forward problem (y, S, z point at per-thread scratch) */
    const double *dy, *dS_T, *dz_T;
    double *dq, *dk, *dvo, *dalpha, *dS0, *dz0;
    size_t next;
    pthread_mutex_t lock;
} bwd_problem;

static double dphi(double x, int kind)
{
    if (kind == OR_PHI_ELU1) return x > 0.0 ? 1.0 : exp(x);
    if (kind == OR_PHI_RELU1) return x > 0.0 ? 1.0 : 0.0;
    return 1.0;
}

/* One forward step on (S, z) in place, exactly as scan_one does it. */
static void fwd_step(const problem *p, size_t bh, int t, double *S, double *z, double *kt)
{
    const int T = p->T, r = p->r, dv = p->dv;
    const size_t row_qk = (bh * (size_t)T + (size_t)t) * (size_t)r;
    const size_t row_v = (bh * (size_t)T + (size_t)t) * (size_t)dv;
    const double a = gate(p, bh, t);
    for (int i = 0; i < r; ++i) kt[i] = phi(decode(p->k, p->in_type, row_qk + i), p->phi_kind);
    for (int i = 0; i < r; ++i) {
        double *Si = S + (size_t)i * dv;
        for (int j = 0; j < dv; ++j) Si[j] = a * Si[j] + kt[i] * decode(p->v, p->in_type, row_v + j);
        z[i] = a * z[i] + kt[i];
    }
}

/* scratch per thread: checkpoints, one segment of states, y, d and vectors */
typedef struct {
    double *ckS, *ckz;         /* [nseg][r*dv], [nseg][r]: state before the segment's first token */
    double *segS, *segz;       /* [kSeg+1][r*dv], [kSeg+1][r]: S_{t0-1} .. S_{t0+kSeg-1} */
    double *y, *d;             /* [T][dv], [T] */
    double *G, *g, *qt, *kt, *dn;
} bwd_scratch;

static void backward_one(const bwd_problem *bp, size_t bh, bwd_scratch *w)
{
    const problem *p = &bp->f;
    const int T = p->T, r = p->r, dv = p->dv;
    const size_t rd = (size_t)r * dv;
    const int nseg = (T + kSeg - 1) / kSeg;

    /* forward sweep: checkpoints, outputs y_t and denominators d_t */
    double *S = w->segS, *z = w->segz;
    if (p->S0) memcpy(S, p->S0 + bh * rd, sizeof(double) * rd);
    else memset(S, 0, sizeof(double) * rd);
    if (p->z0) memcpy(z, p->z0 + bh * (size_t)r, sizeof(double) * (size_t)r);
    else memset(z, 0, sizeof(double) * (size_t)r);
    for (int t = 0; t < T; ++t) {
        if (t % kSeg == 0) {
            memcpy(w->ckS + (size_t)(t / kSeg) * rd, S, sizeof(double) * rd);
            memcpy(w->ckz + (size_t)(t / kSeg) * r, z, sizeof(double) * (size_t)r);
        }
        fwd_step(p, bh, t, S, z, w->kt);
        const size_t row_qk = (bh * (size_t)T + (size_t)t) * (size_t)r;
        for (int i = 0; i < r; ++i) w->qt[i] = phi(decode(p->q, p->in_type, row_qk + i), p->phi_kind);
        double den = 0.0;
        for (int i = 0; i < r; ++i) den += w->qt[i] * z[i];
        den += p->eps;
        w->d[t] = den;
        for (int j = 0; j < dv; ++j) {
            double num = 0.0;
            for (int i = 0; i < r; ++i) num += w->qt[i] * S[(size_t)i * dv + j];
            w->y[(size_t)t * dv + j] = num / den;
        }
    }

    /* reverse sweep */
    double *G = w->G, *g = w->g;
    if (bp->dS_T) memcpy(G, bp->dS_T + bh * rd, sizeof(double) * rd);
    else memset(G, 0, sizeof(double) * rd);
    if (bp->dz_T) memcpy(g, bp->dz_T + bh * (size_t)r, sizeof(double) * (size_t)r);
    else memset(g, 0, sizeof(double) * (size_t)r);
    for (int s = nseg - 1; s >= 0; --s) {
        const int t0 = s * kSeg, t1 = t0 + kSeg < T ? t0 + kSeg : T;
        /* states S_{t0-1} .. S_{t1-1} of this segment, recomputed from its checkpoint */
        memcpy(w->segS, w->ckS + (size_t)s * rd, sizeof(double) * rd);
        memcpy(w->segz, w->ckz + (size_t)s * r, sizeof(double) * (size_t)r);
        for (int t = t0; t < t1; ++t) {
            const int e = t - t0 + 1;
            memcpy(w->segS + (size_t)e * rd, w->segS + (size_t)(e - 1) * rd, sizeof(double) * rd);
            memcpy(w->segz + (size_t)e * r, w->segz + (size_t)(e - 1) * r, sizeof(double) * (size_t)r);
            fwd_step(p, bh, t, w->segS + (size_t)e * rd, w->segz + (size_t)e * r, w->kt);
        }
        for (int t = t1 - 1; t >= t0; --t) {
            const int e = t - t0 + 1;
            const double *St = w->segS + (size_t)e * rd, *Sp = w->segS + (size_t)(e - 1) * rd;
            const double *zt = w->segz + (size_t)e * r, *zp = w->segz + (size_t)(e - 1) * r;
            const size_t row_qk = (bh * (size_t)T + (size_t)t) * (size_t)r;
            const size_t row_v = (bh * (size_t)T + (size_t)t) * (size_t)dv;
            for (int i = 0; i < r; ++i) {
                w->qt[i] = phi(decode(p->q, p->in_type, row_qk + i), p->phi_kind);
                w->kt[i] = phi(decode(p->k, p->in_type, row_qk + i), p->phi_kind);
            }
            /* dn_t = dy_t / d_t, dd_t = -(dy_t . y_t) / d_t */
            double dd = 0.0;
            for (int j = 0; j < dv; ++j) {
                w->dn[j] = bp->dy[row_v + j] / w->d[t];
                dd -= bp->dy[row_v + j] * w->y[(size_t)t * dv + j];
            }
            dd /= w->d[t];
            /* G_t = q~_t dn_t^T + (alpha_{t+1} G_{t+1}),  g_t = dd_t q~_t + (alpha_{t+1} g_{t+1}) */
            for (int i = 0; i < r; ++i) {
                for (int j = 0; j < dv; ++j) G[(size_t)i * dv + j] += w->qt[i] * w->dn[j];
                g[i] += dd * w->qt[i];
            }
            /* dq~_t = S_t dn_t + dd_t z_t ;  dk~_t = G_t v_t + g_t ;  dv_t = G_t^T k~_t */
            for (int i = 0; i < r; ++i) {
                double aq = dd * zt[i], ak = g[i];
                for (int j = 0; j < dv; ++j) {
                    aq += St[(size_t)i * dv + j] * w->dn[j];
                    ak += G[(size_t)i * dv + j] * decode(p->v, p->in_type, row_v + j);
                }
                bp->dq[row_qk + i] = aq * dphi(decode(p->q, p->in_type, row_qk + i), p->phi_kind);
                bp->dk[row_qk + i] = ak * dphi(decode(p->k, p->in_type, row_qk + i), p->phi_kind);
            }
            for (int j = 0; j < dv; ++j) {
                double av = 0.0;
                for (int i = 0; i < r; ++i) av += G[(size_t)i * dv + j] * w->kt[i];
                bp->dvo[row_v + j] = av;
            }
            /* dalpha_t = <G_t, S_{t-1}> + <g_t, z_{t-1}>; then G_{t-1} part: alpha_t G_t */
            const double a = gate(p, bh, t);
            if (p->alpha) {
                double da = 0.0;
                for (size_t x = 0; x < rd; ++x) da += G[x] * Sp[x];
                for (int i = 0; i < r; ++i) da += g[i] * zp[i];
                bp->dalpha[bh * (size_t)T + (size_t)t] = da;
            }
            for (size_t x = 0; x < rd; ++x) G[x] *= a;
            for (int i = 0; i < r; ++i) g[i] *= a;
        }
    }
    memcpy(bp->dS0 + bh * rd, G, sizeof(double) * rd);
    memcpy(bp->dz0 + bh * (size_t)r, g, sizeof(double) * (size_t)r);
}

static void *backward_worker(void *arg)
{
    bwd_problem *bp = (bwd_problem *)arg;
    const problem *p = &bp->f;
    const size_t rd = (size_t)p->r * p->dv, r = (size_t)p->r, dv = (size_t)p->dv, T = (size_t)p->T;
    const size_t nseg = (T + kSeg - 1) / kSeg;
    bwd_scratch w;
    double *buf = (double *)malloc(sizeof(double) * (nseg * (rd + r) + (kSeg + 1) * (rd + r) + T * dv + T +
                                                     rd + 3 * r + dv));
    if (!buf) return NULL;
    w.ckS = buf;
    w.ckz = w.ckS + nseg * rd;
    w.segS = w.ckz + nseg * r;
    w.segz = w.segS + (kSeg + 1) * rd;
    w.y = w.segz + (kSeg + 1) * r;
    w.d = w.y + T * dv;
    w.G = w.d + T;
    w.g = w.G + rd;
    w.qt = w.g + r;
    w.kt = w.qt + r;
    w.dn = w.kt + r;
    const size_t nbh = (size_t)p->B * (size_t)p->H;
    for (;;) {
        pthread_mutex_lock(&bp->lock);
        size_t bh = bp->next++;
        pthread_mutex_unlock(&bp->lock);
        if (bh >= nbh) break;
        backward_one(bp, bh, &w);
    }
    free(buf);
    return NULL;
}

int or_backward(int B, int H, int T, int r, int dv, const void *q, const void *k, const void *v, int in_type,
                const double *alpha, const double *S0, const double *z0, double eps, int phi_kind,
                const double *dy, const double *dS_T, const double *dz_T, int nthreads,
                double *dq, double *dk, double *dvo, double *dalpha, double *dS0, double *dz0)
{
    double dummy = 0.0;
    bwd_problem bp;
    problem f = {B, H, T, r, dv, in_type, phi_kind, 0, q, k, v, alpha, S0, z0, eps, &dummy, &dummy, &dummy};
    if (check(&f)) return -1;
    if (!dy || !dq || !dk || !dvo || !dS0 || !dz0 || (alpha && !dalpha)) return -1;
    bp.f = f;
    bp.dy = dy;
    bp.dS_T = dS_T;
    bp.dz_T = dz_T;
    bp.dq = dq;
    bp.dk = dk;
    bp.dvo = dvo;
    bp.dalpha = dalpha;
    bp.dS0 = dS0;
    bp.dz0 = dz0;
    bp.next = 0;
    pthread_mutex_init(&bp.lock, NULL);
    const size_t nbh = (size_t)B * (size_t)H;
    if (nthreads <= 0) nthreads = or_num_cpus();
    if ((size_t)nthreads > nbh) nthreads = (int)nbh;
    if (nthreads == 1) {
        backward_worker(&bp);
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        if (!th) return -1;
        for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, backward_worker, &bp);
        for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&bp.lock);
    return 0;
}
