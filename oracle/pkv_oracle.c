/*
 * Plain CPU oracle for paged KV-cache decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg load it.  It shares no code, header, table or
 * constant with the CUDA path.
 *
 * What it follows:
 *  - "LLM推論の基礎とvLLMの内部" (ttlab.hopto.org), section 4 "PagedAttention
 *    とブロック管理": K/V live in fixed-size physical blocks (16 tokens by
 *    default); every request keeps a block table from logical to physical
 *    blocks; blocks are filled one at a time; the same prefix may share one
 *    physical block (reference count + copy-on-write).
 *  - the same page, section 2 "KVキャッシュとサイズ式": per-token KV bytes
 *    2 * L * H_kv * d * b; GQA groups query heads onto fewer K/V heads; an
 *    fp8 KV cache stores one byte per element.
 *  - "vLLM 内部構造 (2) — PagedAttention" (youngju.dev), section
 *    "ブロックテーブル": the kernel finds each logical block through the
 *    table; the physical location does not matter.
 *  - section 12 of the first page: PagedAttention is a memory-management
 *    technique, not a different attention, so decode over the paged cache is
 *    textbook softmax attention over the gathered tokens.
 *
 * Every function below is the plain definition written out: gather K/V into
 * contiguous fp64 arrays in logical order, then softmax(scale * q.K^T) V with
 * fp64 accumulation.  No blocking, no fusion, no online softmax.  The
 * optional `partition` argument of the decode computes the same result through
 * per-partition (max, sum, weighted sum) triples and their merge; it exists
 * only so that the merge identity itself can be checked.
 *
 * Number formats are decoded from their definitions:
 *  - fp32 and bf16 (bf16 = the upper 16 bits of an IEEE binary32);
 *  - fp8 E4M3 "fn" of the OCP 8-bit floating point specification: 1 sign
 *    bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
 *    S.1111.111 is NaN, largest finite magnitude 448.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F32 0
#define OR_BF16 1
#define OR_E4M3 2

/* ---------------------------------------------------------------- formats */

/* Value of an E4M3 code, from the OCP definition (sign, biased exponent,
 * mantissa).  Exact in double. */
double oracle_e4m3_to_double(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, 1 - 7);          /* subnormal */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);    /* normal */
    return sign ? -v : v;
}

/* Round |a| (finite, >= 0) to a binary format with `p` significant bits and
 * minimum normal exponent `emin`, round-to-nearest ties-to-even.  The
 * quantum is 2^(max(exponent, emin) - (p-1)); a / quantum is exact in
 * double, and rint() rounds it to the nearest integer with ties to even
 * under the default rounding mode. */
static double round_to_format(double a, int p, int emin)
{
    int E;
    double q;
    if (a == 0.0)
        return 0.0;
    frexp(a, &E);                  /* a = f * 2^E, f in [0.5, 1) */
    E -= 1;                        /* exponent of the leading bit */
    if (E < emin)
        E = emin;
    q = ldexp(1.0, E - (p - 1));
    return rint(a / q) * q;
}

/* float -> E4M3 with round-to-nearest-even and saturation to +-448
 * ("satfinite"); NaN maps to the NaN code.  The rounded magnitude is looked
 * up among the 127 non-negative finite codes (0x00..0x7E), which are in
 * increasing order of value. */
uint8_t oracle_e4m3_from_float(float x)
{
    double a = fabs((double)x);
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double r;
    int c, lo = 0, hi = 0x7E;
    if (isnan(x))
        return (uint8_t)(sign | 0x7F);
    r = round_to_format(a, 4, -6);
    if (r > 448.0)
        r = 448.0;
    /* binary search for the code whose value is exactly r */
    while (lo < hi) {
        c = (lo + hi) / 2;
        if (oracle_e4m3_to_double((uint8_t)c) < r)
            lo = c + 1;
        else
            hi = c;
    }
    return (uint8_t)(sign | lo);
}

double oracle_bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* double -> bf16 (8 significant bits, exponent range of binary32), round to
 * nearest even; overflow past the largest finite value goes to infinity. */
uint16_t oracle_bf16_from_double(double x)
{
    double a = fabs(x), r;
    float f;
    uint32_t u;
    if (isnan(x))
        return 0x7FC0;
    r = round_to_format(a, 8, -126);
    if (r > 3.3895313892515355e38)   /* (2 - 2^-7) * 2^127 */
        r = INFINITY;
    f = (float)(signbit(x) ? -r : r);   /* exact: r has <= 8 significant bits */
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* Element `i` of a raw array of dtype `dt`, as double (fp8 codes are
 * multiplied by `scale`: the stored value is code * scale). */
static double load_elem(const void* base, int dt, size_t i, double scale)
{
    if (dt == OR_F32) {
        float f;
        memcpy(&f, (const char*)base + 4 * i, 4);
        return (double)f;
    }
    if (dt == OR_BF16) {
        uint16_t h;
        memcpy(&h, (const char*)base + 2 * i, 2);
        return oracle_bf16_to_double(h);
    }
    return oracle_e4m3_to_double(((const uint8_t*)base)[i]) * scale;
}

/* ------------------------------------------------------------------ write */

/* reshape_and_cache: token i of `key`/`value` ([T, Hkv, d], dtype in_dt)
 * goes to slot s = slot_mapping[i] of the cache ([NB, bs, Hkv, d], dtype
 * cache_dt): physical block s / bs, offset s % bs.  s < 0 means "no slot"
 * and the token is skipped.
 *   fp32 -> fp32, bf16 -> bf16, bf16 -> fp32: exact.
 *   fp32 -> bf16: round to nearest even.
 *   (fp32 or bf16) -> E4M3: code = e4m3(float(x) / scale), where the divide is
 *   one IEEE binary32 division, rounded to nearest even, saturating.
 * Returns 0, or -1 if a slot is out of range (nothing is written for it). */
int oracle_paged_kv_write(const void* key, const void* value, int in_dt,
                          void* key_cache, void* value_cache, int cache_dt,
                          const int64_t* slot_mapping, int T, int NB, int bs,
                          int Hkv, int d, float k_scale, float v_scale)
{
    int i, h, e, which, bad = 0;
    for (i = 0; i < T; ++i) {
        int64_t s = slot_mapping[i];
        if (s < 0)
            continue;
        if (s >= (int64_t)NB * bs) {
            bad = 1;
            continue;
        }
        for (which = 0; which < 2; ++which) {
            const void* src = which ? value : key;
            void* dst = which ? value_cache : key_cache;
            float sc = which ? v_scale : k_scale;
            for (h = 0; h < Hkv; ++h) {
                for (e = 0; e < d; ++e) {
                    size_t si = ((size_t)i * Hkv + h) * d + e;
                    size_t di = (((size_t)(s / bs) * bs + (size_t)(s % bs)) * Hkv + h) * d + e;
                    double x = load_elem(src, in_dt, si, 1.0);
                    if (cache_dt == OR_F32) {
                        float f = (float)x;   /* exact: x is fp32 or bf16 */
                        memcpy((char*)dst + 4 * di, &f, 4);
                    } else if (cache_dt == OR_BF16) {
                        uint16_t b = oracle_bf16_from_double(x);
                        memcpy((char*)dst + 2 * di, &b, 2);
                    } else {
                        volatile float xf = (float)x;   /* exact */
                        volatile float q = xf / sc;     /* one binary32 divide */
                        ((uint8_t*)dst)[di] = oracle_e4m3_from_float(q);
                    }
                }
            }
        }
    }
    return bad ? -1 : 0;
}

/* ----------------------------------------------------------------- decode */

typedef struct {
    /* inputs */
    const void* q; int q_dt;
    const void* kc; const void* vc; int c_dt;
    const int32_t* block_tables; int MB;
    const int32_t* token_slots; int MT;     /* if set: gather through the token table instead */
    const int32_t* context_lens; int S;
    int Hq, Hkv, d, bs, NB;
    double scale, k_scale, v_scale;
    int partition;          /* 0: one softmax over all tokens */
    /* outputs */
    double* out;            /* [S, Hq, d] */
    /* work split */
    int next;               /* next sequence to take (guarded by mu) */
    pthread_mutex_t mu;
    int status;
} decode_job;

/* Decode one sequence: gather, then the textbook formula per query head. */
static int decode_one(decode_job* J, int s, double* Kc, double* Vc, double* x, double* qh)
{
    int n = J->context_lens[s];
    int g = J->Hq / J->Hkv;
    int t, h, e, kvh;
    double* out = J->out + (size_t)s * J->Hq * J->d;
    if (n < 0 || (J->token_slots ? n > J->MT : n > J->MB * J->bs))
        return -1;
    /* gather K/V of every cached token, in logical order: through the block
     * table (logical block t / bs, offset t % bs), or through the token table
     * (token t sits in slot token_slots[s][t] = block * bs + offset) */
    for (t = 0; t < n; ++t) {
        int pb, off;
        if (J->token_slots) {
            int64_t slot = J->token_slots[(size_t)s * J->MT + t];
            if (slot < 0 || slot >= (int64_t)J->NB * J->bs)
                return -1;
            pb = (int)(slot / J->bs);
            off = (int)(slot % J->bs);
        } else {
            pb = J->block_tables[(size_t)s * J->MB + t / J->bs];
            off = t % J->bs;
        }
        if (pb < 0 || pb >= J->NB)
            return -1;
        for (kvh = 0; kvh < J->Hkv; ++kvh)
            for (e = 0; e < J->d; ++e) {
                size_t src = (((size_t)pb * J->bs + off) * J->Hkv + kvh) * J->d + e;
                size_t dst = ((size_t)t * J->Hkv + kvh) * J->d + e;
                Kc[dst] = load_elem(J->kc, J->c_dt, src, J->k_scale);
                Vc[dst] = load_elem(J->vc, J->c_dt, src, J->v_scale);
            }
    }
    for (h = 0; h < J->Hq; ++h) {
        double* o = out + (size_t)h * J->d;
        kvh = h / g;                      /* contiguous GQA grouping */
        for (e = 0; e < J->d; ++e)
            o[e] = 0.0;
        if (n == 0)
            continue;
        /* logits x_t = scale * <q_h, k_t> */
        for (e = 0; e < J->d; ++e)
            qh[e] = load_elem(J->q, J->q_dt, ((size_t)s * J->Hq + h) * J->d + e, 1.0);
        for (t = 0; t < n; ++t) {
            double acc = 0.0;
            for (e = 0; e < J->d; ++e)
                acc += qh[e] * Kc[((size_t)t * J->Hkv + kvh) * J->d + e];
            x[t] = J->scale * acc;
        }
        if (J->partition <= 0) {
            double m = -INFINITY, l = 0.0;
            for (t = 0; t < n; ++t)
                if (x[t] > m)
                    m = x[t];
            for (t = 0; t < n; ++t) {
                double p = exp(x[t] - m);
                l += p;
                for (e = 0; e < J->d; ++e)
                    o[e] += p * Vc[((size_t)t * J->Hkv + kvh) * J->d + e];
            }
            for (e = 0; e < J->d; ++e)
                o[e] /= l;
        } else {
            /* Split form: each partition of `partition` tokens yields its own
             * (m_p, l_p, acc_p); the merge takes M = max m_p,
             * L = sum e^(m_p - M) l_p, O = sum e^(m_p - M) acc_p / L. */
            int P = J->partition, np = (n + P - 1) / P, p;
            double M = -INFINITY, L = 0.0;
            double* mp = malloc(sizeof(double) * np);
            double* lp = malloc(sizeof(double) * np);
            double* ap = calloc((size_t)np * J->d, sizeof(double));
            if (!mp || !lp || !ap) {
                free(mp); free(lp); free(ap);
                return -2;
            }
            for (p = 0; p < np; ++p) {
                int t0 = p * P, t1 = t0 + P < n ? t0 + P : n;
                mp[p] = -INFINITY;
                lp[p] = 0.0;
                for (t = t0; t < t1; ++t)
                    if (x[t] > mp[p])
                        mp[p] = x[t];
                for (t = t0; t < t1; ++t) {
                    double w = exp(x[t] - mp[p]);
                    lp[p] += w;
                    for (e = 0; e < J->d; ++e)
                        ap[(size_t)p * J->d + e] += w * Vc[((size_t)t * J->Hkv + kvh) * J->d + e];
                }
                if (mp[p] > M)
                    M = mp[p];
            }
            for (p = 0; p < np; ++p) {
                double w = exp(mp[p] - M);
                L += w * lp[p];
                for (e = 0; e < J->d; ++e)
                    o[e] += w * ap[(size_t)p * J->d + e];
            }
            for (e = 0; e < J->d; ++e)
                o[e] /= L;
            free(mp); free(lp); free(ap);
        }
    }
    return 0;
}

static void* decode_worker(void* arg)
{
    decode_job* J = (decode_job*)arg;
    size_t maxtok = J->token_slots ? (size_t)J->MT : (size_t)J->MB * J->bs;
    double* Kc = malloc(sizeof(double) * (maxtok ? maxtok : 1) * J->Hkv * J->d);
    double* Vc = malloc(sizeof(double) * (maxtok ? maxtok : 1) * J->Hkv * J->d);
    double* x = malloc(sizeof(double) * (maxtok ? maxtok : 1));
    double* qh = malloc(sizeof(double) * J->d);
    if (!Kc || !Vc || !x || !qh) {
        pthread_mutex_lock(&J->mu);
        J->status = -2;
        pthread_mutex_unlock(&J->mu);
    } else {
        for (;;) {
            int s, rc;
            pthread_mutex_lock(&J->mu);
            s = J->next++;
            pthread_mutex_unlock(&J->mu);
            if (s >= J->S)
                break;
            rc = decode_one(J, s, Kc, Vc, x, qh);
            if (rc) {
                pthread_mutex_lock(&J->mu);
                J->status = rc;
                pthread_mutex_unlock(&J->mu);
            }
        }
    }
    free(Kc); free(Vc); free(x); free(qh);
    return NULL;
}

/* Paged decode attention.  q: [S, Hq, d] (fp32 or bf16); caches
 * [NB, bs, Hkv, d] (fp32, bf16 or E4M3 codes with dequantised value
 * code * k_scale / code * v_scale); block_tables int32 [S, MB];
 * context_lens int32 [S].  out: fp64 [S, Hq, d].  A sequence with no
 * tokens gives zeros.  partition > 0 computes the same result through
 * per-partition (max, sum, weighted sum) triples and their merge.  Runs
 * `threads` POSIX threads over sequences.  Returns 0, -1 on an
 * out-of-range block id or length, -2 on allocation failure. */
static int run_decode(double* out, const void* q, int q_dt, const void* key_cache, const void* value_cache,
                      int cache_dt, const int32_t* block_tables, int MB, const int32_t* token_slots, int MT,
                      const int32_t* context_lens, int S, int Hq, int Hkv, int d, int bs, int NB, float scale,
                      float k_scale, float v_scale, int partition, int threads)
{
    decode_job J;
    pthread_t* tid;
    int i, nt = threads > 0 ? threads : 1;
    if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || bs <= 0)
        return -1;
    memset(&J, 0, sizeof J);
    J.q = q; J.q_dt = q_dt; J.kc = key_cache; J.vc = value_cache; J.c_dt = cache_dt;
    J.block_tables = block_tables; J.MB = MB; J.token_slots = token_slots; J.MT = MT;
    J.context_lens = context_lens; J.S = S;
    J.Hq = Hq; J.Hkv = Hkv; J.d = d; J.bs = bs; J.NB = NB;
    J.scale = (double)scale;
    J.k_scale = cache_dt == OR_E4M3 ? (double)k_scale : 1.0;
    J.v_scale = cache_dt == OR_E4M3 ? (double)v_scale : 1.0;
    J.partition = partition; J.out = out;
    pthread_mutex_init(&J.mu, NULL);
    if (nt > S)
        nt = S > 0 ? S : 1;
    tid = malloc(sizeof(pthread_t) * nt);
    if (!tid)
        return -2;
    for (i = 0; i < nt; ++i)
        pthread_create(&tid[i], NULL, decode_worker, &J);
    for (i = 0; i < nt; ++i)
        pthread_join(tid[i], NULL);
    free(tid);
    pthread_mutex_destroy(&J.mu);
    return J.status;
}

int oracle_paged_attention_decode(double* out, const void* q, int q_dt,
                                  const void* key_cache, const void* value_cache,
                                  int cache_dt, const int32_t* block_tables, int MB,
                                  const int32_t* context_lens, int S, int Hq, int Hkv,
                                  int d, int bs, int NB, float scale, float k_scale,
                                  float v_scale, int partition, int threads)
{
    return run_decode(out, q, q_dt, key_cache, value_cache, cache_dt, block_tables, MB, NULL, 0, context_lens, S,
                      Hq, Hkv, d, bs, NB, scale, k_scale, v_scale, partition, threads);
}

/* ---------------------------------------------------------------- prefill */

typedef struct {
    decode_job base;                /* caches, tables, lengths, sizes */
    const int32_t* query_start;     /* [S + 1] */
} prefill_job;

/* Several query tokens per sequence (a prefill chunk, or tokens proposed by
 * speculative decoding): the sequence's last q_len = query_start[s+1] -
 * query_start[s] tokens are the queries, their K/V already in the cache.
 * Query i sits at position p = n - q_len + i and attends to tokens 0..p
 * (causal).  Same gather-then-textbook-softmax as the decode. */
static int prefill_one(prefill_job* P, int s, double* Kc, double* Vc, double* x, double* qh)
{
    decode_job* J = &P->base;
    int n = J->context_lens[s];
    int q0 = P->query_start[s], ql = P->query_start[s + 1] - q0;
    int g = J->Hq / J->Hkv;
    int t, h, e, kvh, i;
    if (n < 0 || n > J->MB * J->bs || ql < 0 || ql > n)
        return -1;
    for (t = 0; t < n; ++t) {
        int pb = J->block_tables[(size_t)s * J->MB + t / J->bs];
        int off = t % J->bs;
        if (pb < 0 || pb >= J->NB)
            return -1;
        for (kvh = 0; kvh < J->Hkv; ++kvh)
            for (e = 0; e < J->d; ++e) {
                size_t src = (((size_t)pb * J->bs + off) * J->Hkv + kvh) * J->d + e;
                size_t dst = ((size_t)t * J->Hkv + kvh) * J->d + e;
                Kc[dst] = load_elem(J->kc, J->c_dt, src, J->k_scale);
                Vc[dst] = load_elem(J->vc, J->c_dt, src, J->v_scale);
            }
    }
    for (i = 0; i < ql; ++i) {
        int pos = n - ql + i;
        for (h = 0; h < J->Hq; ++h) {
            double* o = J->out + ((size_t)(q0 + i) * J->Hq + h) * J->d;
            double m = -INFINITY, l = 0.0;
            kvh = h / g;
            for (e = 0; e < J->d; ++e) {
                qh[e] = load_elem(J->q, J->q_dt, ((size_t)(q0 + i) * J->Hq + h) * J->d + e, 1.0);
                o[e] = 0.0;
            }
            for (t = 0; t <= pos; ++t) {
                double acc = 0.0;
                for (e = 0; e < J->d; ++e)
                    acc += qh[e] * Kc[((size_t)t * J->Hkv + kvh) * J->d + e];
                x[t] = J->scale * acc;
                if (x[t] > m)
                    m = x[t];
            }
            for (t = 0; t <= pos; ++t) {
                double p = exp(x[t] - m);
                l += p;
                for (e = 0; e < J->d; ++e)
                    o[e] += p * Vc[((size_t)t * J->Hkv + kvh) * J->d + e];
            }
            for (e = 0; e < J->d; ++e)
                o[e] /= l;
        }
    }
    return 0;
}

static void* prefill_worker(void* arg)
{
    prefill_job* P = (prefill_job*)arg;
    decode_job* J = &P->base;
    size_t maxtok = (size_t)J->MB * J->bs;
    double* Kc = malloc(sizeof(double) * (maxtok ? maxtok : 1) * J->Hkv * J->d);
    double* Vc = malloc(sizeof(double) * (maxtok ? maxtok : 1) * J->Hkv * J->d);
    double* x = malloc(sizeof(double) * (maxtok ? maxtok : 1));
    double* qh = malloc(sizeof(double) * J->d);
    if (!Kc || !Vc || !x || !qh) {
        pthread_mutex_lock(&J->mu);
        J->status = -2;
        pthread_mutex_unlock(&J->mu);
    } else {
        for (;;) {
            int s, rc;
            pthread_mutex_lock(&J->mu);
            s = J->next++;
            pthread_mutex_unlock(&J->mu);
            if (s >= J->S)
                break;
            rc = prefill_one(P, s, Kc, Vc, x, qh);
            if (rc) {
                pthread_mutex_lock(&J->mu);
                J->status = rc;
                pthread_mutex_unlock(&J->mu);
            }
        }
    }
    free(Kc); free(Vc); free(x); free(qh);
    return NULL;
}

/* out: fp64 [T, Hq, d] with T = query_start[S]; q: [T, Hq, d]. */
int oracle_paged_attention_prefill(double* out, const void* q, int q_dt, const void* key_cache,
                                   const void* value_cache, int cache_dt, const int32_t* block_tables,
                                   int MB, const int32_t* context_lens, const int32_t* query_start, int S,
                                   int Hq, int Hkv, int d, int bs, int NB, float scale, float k_scale,
                                   float v_scale, int threads)
{
    prefill_job P;
    pthread_t* tid;
    int i, nt = threads > 0 ? threads : 1;
    if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || bs <= 0)
        return -1;
    memset(&P, 0, sizeof P);
    P.base.q = q; P.base.q_dt = q_dt; P.base.kc = key_cache; P.base.vc = value_cache;
    P.base.c_dt = cache_dt; P.base.block_tables = block_tables; P.base.MB = MB;
    P.base.context_lens = context_lens; P.base.S = S; P.base.Hq = Hq; P.base.Hkv = Hkv;
    P.base.d = d; P.base.bs = bs; P.base.NB = NB; P.base.scale = (double)scale;
    P.base.k_scale = cache_dt == OR_E4M3 ? (double)k_scale : 1.0;
    P.base.v_scale = cache_dt == OR_E4M3 ? (double)v_scale : 1.0;
    P.base.out = out;
    P.query_start = query_start;
    pthread_mutex_init(&P.base.mu, NULL);
    if (nt > S)
        nt = S > 0 ? S : 1;
    tid = malloc(sizeof(pthread_t) * nt);
    if (!tid)
        return -2;
    for (i = 0; i < nt; ++i)
        pthread_create(&tid[i], NULL, prefill_worker, &P);
    for (i = 0; i < nt; ++i)
        pthread_join(tid[i], NULL);
    free(tid);
    pthread_mutex_destroy(&P.base.mu);
    return P.base.status;
}

/* ------------------------------------------------------------ copy_blocks */

/* Copy-on-write duplication: for every layer and every (src, dst) pair of
 * block_mapping ([P, 2]), physical block dst of the K and V caches becomes a
 * byte copy of block src.  block_bytes = bs * Hkv * d * element size.
 * Returns 0, or -1 if a block id is out of range (that pair is skipped). */
int oracle_copy_blocks(void* const* key_caches, void* const* value_caches, int num_layers,
                       const int64_t* block_mapping, int P, int NB, size_t block_bytes)
{
    int l, p, bad = 0;
    for (l = 0; l < num_layers; ++l)
        for (p = 0; p < P; ++p) {
            int64_t src = block_mapping[2 * p], dst = block_mapping[2 * p + 1];
            if (src < 0 || src >= NB || dst < 0 || dst >= NB) {
                bad = 1;
                continue;
            }
            memcpy((char*)key_caches[l] + dst * block_bytes,
                   (const char*)key_caches[l] + src * block_bytes, block_bytes);
            memcpy((char*)value_caches[l] + dst * block_bytes,
                   (const char*)value_caches[l] + src * block_bytes, block_bytes);
        }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------ token table */

/*
 * Decode attention through a token table ("LLM推論の「見えないメモリ問題」を
 * 解く … vToken", section on token-level virtualisation): the table maps each
 * live token, in the sequence's logical order, to its physical slot
 * block * bs + offset; deleted tokens are simply absent.  The result is the
 * textbook softmax attention over the live tokens, as in the decode above.
 * token_slots [S, MT]; num_tokens [S] live tokens per sequence.
 */
int oracle_token_attention_decode(double* out, const void* q, int q_dt, const void* key_cache,
                                  const void* value_cache, int cache_dt, const int32_t* token_slots, int MT,
                                  const int32_t* num_tokens, int S, int Hq, int Hkv, int d, int bs, int NB,
                                  float scale, float k_scale, float v_scale, int threads)
{
    return run_decode(out, q, q_dt, key_cache, value_cache, cache_dt, NULL, 0, token_slots, MT, num_tokens, S,
                      Hq, Hkv, d, bs, NB, scale, k_scale, v_scale, 0, threads);
}

/*
 * Repacking (same page, "非同期リパッキング"): live tokens move to free slots
 * of other blocks so that emptied blocks can be released; the token table
 * entry of each moved token is rewritten, and the logical order is kept.
 * moves [M, 4] = (sequence, logical index, source slot, destination slot);
 * a move applies only if its indices are in range and the table holds the
 * source slot at that position.  Every layer's K and V row of the token
 * (token_bytes bytes each) is copied.  Returns -1 if any move was skipped.
 */
int oracle_repack_tokens(void* const* key_caches, void* const* value_caches, int num_layers, int32_t* token_slots,
                         int MT, int S, const int64_t* moves, int M, int NB, int bs, size_t token_bytes)
{
    int i, l, bad = 0;
    const int64_t slots = (int64_t)NB * bs;
    for (i = 0; i < M; ++i) {
        int64_t seq = moves[4 * i], idx = moves[4 * i + 1], src = moves[4 * i + 2], dst = moves[4 * i + 3];
        if (seq < 0 || seq >= S || idx < 0 || idx >= MT || src < 0 || src >= slots || dst < 0 || dst >= slots ||
            token_slots[seq * MT + idx] != src) {
            bad = 1;
            continue;
        }
        for (l = 0; l < num_layers; ++l) {
            memcpy((char*)key_caches[l] + dst * token_bytes, (const char*)key_caches[l] + src * token_bytes,
                   token_bytes);
            memcpy((char*)value_caches[l] + dst * token_bytes, (const char*)value_caches[l] + src * token_bytes,
                   token_bytes);
        }
        token_slots[seq * MT + idx] = (int32_t)dst;
    }
    return bad ? -1 : 0;
}

/* --------------------------------------------------------- byte accounting */

/* Bytes of K and V one token occupies across all layers: 2 * L * H_kv * d * b
 * (first page, section 2). */
long long oracle_kv_bytes_per_token(int L, int Hkv, int d, int b)
{
    return 2LL * L * Hkv * d * b;
}

/* Physical blocks a sequence of n tokens holds: ceil(n / bs) (first page,
 * section 4: blocks are handed out one at a time as tokens arrive). */
long long oracle_blocks_for_tokens(long long n, int bs)
{
    return (n + bs - 1) / bs;
}
