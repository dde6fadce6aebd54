/*
 * oracle.c -- plain, slow, obviously correct CPU oracle for the DDTree
 * tree-verify step.  TEST INFRASTRUCTURE ONLY: see oracle.h for what it
 * computes, where each part comes from on the pages, its layouts and its
 * precision.  No blocking, fusion or reordering beyond the definitions.
 */
#ifdef _OPENMP
#include <omp.h>
#endif
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* scalar conversions                                                        */
/* ------------------------------------------------------------------------ */

double orc_bf16_to_double(uint16_t h) {
    /* bf16 is the top half of an IEEE binary32. */
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

float orc_half_to_float(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);                 /* zero or subnormal */
    } else if (e == 31) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexp(1.0 + (double)m / 1024.0, e - 15);
    }
    return (float)(sign ? -v : v);
}

uint16_t orc_float_to_half_rn(float f) {
    /* IEEE binary16, round to nearest, ties to even.  Every intermediate
     * below is exact in double, and rint() rounds ties to even. */
    if (isnan(f)) return 0x7e00;
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    double a = fabs((double)f);
    if (a >= 65520.0) return sign | 0x7c00;         /* rounds past 65504 */
    if (a < ldexp(1.0, -14)) {                       /* subnormal range */
        double m = rint(a / ldexp(1.0, -24));        /* 0 .. 1024 */
        return sign | (uint16_t)m;                   /* 1024 = smallest normal */
    }
    int e2;
    double fr = frexp(a, &e2);                       /* a = fr * 2^e2, fr in [0.5,1) */
    int E = e2 - 1;                                  /* a = (2 fr) * 2^E */
    double m = rint((2.0 * fr - 1.0) * 1024.0);      /* 0 .. 1024 */
    if (m >= 1024.0) { m = 0.0; E += 1; }
    if (E + 15 >= 31) return sign | 0x7c00;
    return sign | (uint16_t)(((E + 15) << 10) | (int)m);
}

/* ------------------------------------------------------------------------ */
/* tree topology                                                             */
/* ------------------------------------------------------------------------ */

int orc_tree_topology(int n, const int32_t* parent, int32_t* depth, uint64_t* anc_self) {
    /* Node 0 is the root (the last committed token); every other node's
     * parent precedes it, so the parent array is in topological order. */
    if (n < 1 || n > 64) return ORC_ERR_TOPOLOGY;
    if (parent[0] != -1) return ORC_ERR_TOPOLOGY;
    depth[0] = 0;
    anc_self[0] = 1ull;
    for (int i = 1; i < n; ++i) {
        int p = parent[i];
        if (p < 0 || p >= i) return ORC_ERR_TOPOLOGY;
        depth[i] = depth[p] + 1;
        anc_self[i] = anc_self[p] | (1ull << i);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* gated delta rule                                                          */
/* ------------------------------------------------------------------------ */

void orc_gdn_step(int dv, int dk, const double* S, const double* q, const double* k,
                  const double* v, double beta, double alpha, double* S_out, double* o) {
    /* S_out = alpha * S (I - beta k k^T) + beta v k^T, written per element:
     *   (S (I - beta k k^T))[r][c] = S[r][c] - beta * (sum_c' S[r][c'] k[c']) * k[c]. */
    for (int r = 0; r < dv; ++r) {
        const double* Sr = S + (size_t)r * dk;
        double* Or = S_out + (size_t)r * dk;
        double sk = 0.0;
        for (int c = 0; c < dk; ++c) sk += Sr[c] * k[c];
        for (int c = 0; c < dk; ++c)
            Or[c] = alpha * (Sr[c] - beta * sk * k[c]) + beta * v[r] * k[c];
    }
    /* o = S_out q: the output reads the updated state. */
    for (int r = 0; r < dv; ++r) {
        const double* Or = S_out + (size_t)r * dk;
        double acc = 0.0;
        for (int c = 0; c < dk; ++c) acc += Or[c] * q[c];
        o[r] = acc;
    }
}

typedef struct {
    int B, N, Hk, Hv, dk, dv;
    const uint16_t *q, *k, *v;
    const float *beta, *log_alpha;
} gdn_inputs;

/* Loads node i's inputs for v-head h.  q/k head = h / (Hv / Hk): the v-heads
 * are grouped contiguously over the q/k heads. */
static void gdn_node_inputs(const gdn_inputs* in, int b, int i, int h,
                            double* q, double* k, double* v, double* beta, double* alpha) {
    int hk = h / (in->Hv / in->Hk);
    size_t qk_off = (((size_t)b * in->N + i) * in->Hk + hk) * in->dk;
    size_t v_off = (((size_t)b * in->N + i) * in->Hv + h) * in->dv;
    size_t s_off = ((size_t)b * in->N + i) * in->Hv + h;
    for (int c = 0; c < in->dk; ++c) {
        q[c] = orc_bf16_to_double(in->q[qk_off + c]);
        k[c] = orc_bf16_to_double(in->k[qk_off + c]);
    }
    for (int r = 0; r < in->dv; ++r) v[r] = orc_bf16_to_double(in->v[v_off + r]);
    *beta = (double)in->beta[s_off];
    *alpha = exp((double)in->log_alpha[s_off]);
}

static int gdn_dims_ok(int B, int N, int Hk, int Hv, int dk, int dv) {
    return B >= 1 && N >= 1 && N <= 64 && Hk >= 1 && Hv >= Hk && Hv % Hk == 0 && dk >= 1 && dv >= 1;
}

int orc_tree_gdn_verify(int B, int N, int Hk, int Hv, int dk, int dv,
                        const int32_t* parent, const int32_t* n_nodes,
                        const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const float* beta, const float* log_alpha, const float* state,
                        float* out, double* node_states) {
    if (!gdn_dims_ok(B, N, Hk, Hv, dk, dv)) return ORC_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        int32_t depth[64];
        uint64_t anc[64];
        if (n_nodes[b] > N || orc_tree_topology(n_nodes[b], parent + (size_t)b * N, depth, anc) != ORC_OK)
            return ORC_ERR_TOPOLOGY;
    }
    gdn_inputs in = {B, N, Hk, Hv, dk, dv, q, k, v, beta, log_alpha};
    const size_t SS = (size_t)dv * dk;
    /* every (sequence, head) is independent: the same steps in the same
     * order whichever thread takes it */
#pragma omp parallel
    {
        double* S0 = malloc(SS * sizeof(double));
        double* states = malloc((size_t)N * SS * sizeof(double));
        double *qd = malloc(dk * sizeof(double)), *kd = malloc(dk * sizeof(double));
        double *vd = malloc(dv * sizeof(double)), *od = malloc(dv * sizeof(double));
#pragma omp for schedule(dynamic)
        for (int bh = 0; bh < B * Hv; ++bh) {
            const int b = bh / Hv, h = bh % Hv, n = n_nodes[b];
            const float* Sf = state + ((size_t)b * Hv + h) * SS;
            for (size_t e = 0; e < SS; ++e) S0[e] = (double)Sf[e];
            for (int i = 0; i < n; ++i) {
                int p = parent[(size_t)b * N + i];
                const double* Sp = (p < 0) ? S0 : states + (size_t)p * SS;
                double be, al;
                gdn_node_inputs(&in, b, i, h, qd, kd, vd, &be, &al);
                orc_gdn_step(dv, dk, Sp, qd, kd, vd, be, al, states + (size_t)i * SS, od);
                float* o = out + (((size_t)b * N + i) * Hv + h) * dv;
                for (int r = 0; r < dv; ++r) o[r] = (float)od[r];
                if (node_states)
                    memcpy(node_states + (((size_t)b * N + i) * Hv + h) * SS,
                           states + (size_t)i * SS, SS * sizeof(double));
            }
        }
        free(S0); free(states); free(qd); free(kd); free(vd); free(od);
    }
    return ORC_OK;
}

int orc_tree_gdn_verify_bruteforce(int B, int N, int Hk, int Hv, int dk, int dv,
                                   const int32_t* parent, const int32_t* n_nodes,
                                   const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                   const float* beta, const float* log_alpha,
                                   const float* state, float* out) {
    if (!gdn_dims_ok(B, N, Hk, Hv, dk, dv)) return ORC_ERR_ARG;
    gdn_inputs in = {B, N, Hk, Hv, dk, dv, q, k, v, beta, log_alpha};
    size_t SS = (size_t)dv * dk;
    double* Sa = malloc(SS * sizeof(double));
    double* Sb = malloc(SS * sizeof(double));
    double *qd = malloc(dk * sizeof(double)), *kd = malloc(dk * sizeof(double));
    double *vd = malloc(dv * sizeof(double)), *od = malloc(dv * sizeof(double));
    int rc = ORC_OK;
    for (int b = 0; b < B && rc == ORC_OK; ++b) {
        int n = n_nodes[b];
        int32_t depth[64];
        uint64_t anc[64];
        if (n > N || orc_tree_topology(n, parent + (size_t)b * N, depth, anc) != ORC_OK) {
            rc = ORC_ERR_TOPOLOGY;
            break;
        }
        for (int h = 0; h < Hv; ++h) {
            for (int i = 0; i < n; ++i) {
                /* the root-to-i path, root first */
                int path[64], len = 0;
                for (int c = i; c >= 0; c = parent[(size_t)b * N + c]) path[len++] = c;
                const float* Sf = state + ((size_t)b * Hv + h) * SS;
                for (size_t e = 0; e < SS; ++e) Sa[e] = (double)Sf[e];
                for (int m = len - 1; m >= 0; --m) {
                    double be, al;
                    gdn_node_inputs(&in, b, path[m], h, qd, kd, vd, &be, &al);
                    orc_gdn_step(dv, dk, Sa, qd, kd, vd, be, al, Sb, od);
                    double* t = Sa; Sa = Sb; Sb = t;
                }
                float* o = out + (((size_t)b * N + i) * Hv + h) * dv;
                for (int r = 0; r < dv; ++r) o[r] = (float)od[r];
            }
        }
    }
    free(Sa); free(Sb); free(qd); free(kd); free(vd); free(od);
    return rc;
}

int orc_gdn_commit(int B, int N, int Hk, int Hv, int dk, int dv,
                   const uint16_t* q, const uint16_t* k, const uint16_t* v,
                   const float* beta, const float* log_alpha,
                   const int32_t* path, const int32_t* path_len, float* state) {
    if (!gdn_dims_ok(B, N, Hk, Hv, dk, dv)) return ORC_ERR_ARG;
    gdn_inputs in = {B, N, Hk, Hv, dk, dv, q, k, v, beta, log_alpha};
    const size_t SS = (size_t)dv * dk;
    for (int b = 0; b < B; ++b)
        if (path_len[b] < 1 || path_len[b] > N) return ORC_ERR_ARG;
#pragma omp parallel
    {
        double* Sa = malloc(SS * sizeof(double));
        double* Sb = malloc(SS * sizeof(double));
        double *qd = malloc(dk * sizeof(double)), *kd = malloc(dk * sizeof(double));
        double *vd = malloc(dv * sizeof(double)), *od = malloc(dv * sizeof(double));
#pragma omp for schedule(dynamic)
        for (int bh = 0; bh < B * Hv; ++bh) {
            const int b = bh / Hv, h = bh % Hv, L = path_len[b];
            float* Sf = state + ((size_t)b * Hv + h) * SS;
            for (size_t e = 0; e < SS; ++e) Sa[e] = (double)Sf[e];
            /* decode exactly the accepted tokens, in path order */
            for (int m = 0; m < L; ++m) {
                double be, al;
                gdn_node_inputs(&in, b, path[(size_t)b * N + m], h, qd, kd, vd, &be, &al);
                orc_gdn_step(dv, dk, Sa, qd, kd, vd, be, al, Sb, od);
                double* t = Sa; Sa = Sb; Sb = t;
            }
            for (size_t e = 0; e < SS; ++e) Sf[e] = (float)Sa[e];
        }
        free(Sa); free(Sb); free(qd); free(kd); free(vd); free(od);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* block quantisation: 32 values sharing one fp16 scale d                    */
/* ------------------------------------------------------------------------ */

/* q8_0: d = amax / 127 (stored as fp16), codes = clamp(round_half_away(x * (1/d)), -127, 127)
 * with the reciprocal taken of the fp32 d: the format's usual quantiser. */
void orc_quantize_q8_0(const float* x, int8_t* qs, uint16_t* d16) {
    float amax = 0.0f;
    for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(x[j]));
    float d = amax / 127.0f;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    *d16 = orc_float_to_half_rn(d);
    for (int j = 0; j < 32; ++j) {
        float r = roundf(x[j] * id);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        qs[j] = (int8_t)r;
    }
}

/* q4_0: d = amax / 7 (stored as fp16), code = clamp(round_half_away(x * (1/d)), -8, 7) + 8.
 * Element j < 16 sits in the low nibble of byte j, element j + 16 in its
 * high nibble. */
void orc_quantize_q4_0(const float* x, uint8_t* nib, uint16_t* d16) {
    float amax = 0.0f;
    for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(x[j]));
    float d = amax / 7.0f;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    *d16 = orc_float_to_half_rn(d);
    uint8_t code[32];
    for (int j = 0; j < 32; ++j) {
        float r = roundf(x[j] * id);
        if (r > 7.0f) r = 7.0f;
        if (r < -8.0f) r = -8.0f;
        code[j] = (uint8_t)((int)r + 8);
    }
    for (int j = 0; j < 16; ++j) nib[j] = (uint8_t)(code[j] | (code[j + 16] << 4));
}

void orc_dequantize_q8_0(const int8_t* qs, uint16_t d16, double* x) {
    double d = (double)orc_half_to_float(d16);
    for (int j = 0; j < 32; ++j) x[j] = d * (double)qs[j];
}

void orc_dequantize_q4_0(const uint8_t* nib, uint16_t d16, double* x) {
    double d = (double)orc_half_to_float(d16);
    for (int j = 0; j < 16; ++j) {
        x[j] = d * (double)((int)(nib[j] & 0x0f) - 8);
        x[j + 16] = d * (double)((int)(nib[j] >> 4) - 8);
    }
}

/* TQ3_0 (readings in oracle.h): d = amax / 3, three-bit codes packed as a
 * little-endian bit stream, the same rounding as q8_0 / q4_0. */
void orc_quantize_tq3_0(const float* x, uint8_t* codes, uint16_t* d16) {
    float amax = 0.0f;
    for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(x[j]));
    float d = amax / 3.0f;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    *d16 = orc_float_to_half_rn(d);
    for (int j = 0; j < 12; ++j) codes[j] = 0;
    for (int j = 0; j < 32; ++j) {
        float r = roundf(x[j] * id);
        if (r > 3.0f) r = 3.0f;
        if (r < -4.0f) r = -4.0f;
        unsigned c = (unsigned)((int)r + 4);
        int bit = 3 * j;
        codes[bit / 8] |= (uint8_t)(c << (bit % 8));
        if (bit % 8 > 5) codes[bit / 8 + 1] |= (uint8_t)(c >> (8 - bit % 8));
    }
}

void orc_dequantize_tq3_0(const uint8_t* codes, uint16_t d16, double* x) {
    double d = (double)orc_half_to_float(d16);
    for (int j = 0; j < 32; ++j) {
        int bit = 3 * j;
        unsigned v = codes[bit / 8];
        if (bit / 8 + 1 < 12) v |= (unsigned)codes[bit / 8 + 1] << 8;
        int c = (int)((v >> (bit % 8)) & 7u);
        x[j] = d * (double)(c - 4);
    }
}

void orc_fwht_f32(int n, float* x) {
    for (int h = 1; h < n; h *= 2)
        for (int i = 0; i < n; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                float a = x[j], b = x[j + h];
                x[j] = a + b;
                x[j + h] = a - b;
            }
    const float s = (float)(1.0 / sqrt((double)n));
    for (int j = 0; j < n; ++j) x[j] *= s;
}

/* The same transform in fp64, for the query and the output (no integer
 * depends on them). */
static void fwht_f64(int n, double* x) {
    for (int h = 1; h < n; h *= 2)
        for (int i = 0; i < n; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                double a = x[j], b = x[j + h];
                x[j] = a + b;
                x[j + h] = a - b;
            }
    const double s = 1.0 / sqrt((double)n);
    for (int j = 0; j < n; ++j) x[j] *= s;
}

/* ------------------------------------------------------------------------ */
/* attention tree verify                                                     */
/* ------------------------------------------------------------------------ */

typedef struct {
    int B, Hkv, D, cap, type;
    void *kq, *vq;
    uint16_t *ks, *vs;
} kv_cache;

/* The format of one plane (which = 0: keys, 1: values) of a cache type: the
 * asymmetric types quantise keys and values differently ("Luce DFlash"
 * README, "Asymmetric K/V quantization"). */
static int plane_type(int type, int which) {
    if (type == ORC_KV_Q8_0_Q4_0) return which ? ORC_KV_Q4_0 : ORC_KV_Q8_0;
    if (type == ORC_KV_Q4_0_Q8_0) return which ? ORC_KV_Q8_0 : ORC_KV_Q4_0;
    return type;
}

static size_t kv_row_bytes(int type, int D) {
    return type == ORC_KV_Q8_0 ? (size_t)D : type == ORC_KV_Q4_0 ? (size_t)D / 2
           : type == ORC_KV_TQ3_0 ? (size_t)D / 32 * 12 : (size_t)D * 4;
}

/* Keys stored as TQ3_0 put the whole attention in the rotated basis. */
static int kv_rotated(int type) { return type == ORC_KV_TQ3_0; }

static size_t kv_row_index(const kv_cache* c, int b, int h, int pos) {
    return ((size_t)b * c->Hkv + h) * c->cap + pos;
}

/* Dequantises the key (which = 0) or value (which = 1) row at cache slot pos. */
static void kv_read_row(const kv_cache* c, int which, int b, int h, int pos, double* x) {
    size_t row = kv_row_index(c, b, h, pos);
    const uint8_t* plane = (const uint8_t*)(which ? c->vq : c->kq);
    const uint16_t* sc = which ? c->vs : c->ks;
    const int type = plane_type(c->type, which);
    const uint8_t* qrow = plane + row * kv_row_bytes(type, c->D);
    if (type == ORC_KV_F32) {
        const float* f = (const float*)qrow;
        for (int d = 0; d < c->D; ++d) x[d] = (double)f[d];
        return;
    }
    const uint16_t* srow = sc + row * (c->D / 32);
    for (int blk = 0; blk < c->D / 32; ++blk) {
        if (type == ORC_KV_Q8_0)
            orc_dequantize_q8_0((const int8_t*)qrow + 32 * blk, srow[blk], x + 32 * blk);
        else if (type == ORC_KV_TQ3_0)
            orc_dequantize_tq3_0(qrow + 12 * blk, srow[blk], x + 32 * blk);
        else
            orc_dequantize_q4_0(qrow + 16 * blk, srow[blk], x + 32 * blk);
    }
}

/* Quantises one bf16 row into cache slot pos. */
static void kv_write_row(kv_cache* c, int which, int b, int h, int pos, const uint16_t* src) {
    size_t row = kv_row_index(c, b, h, pos);
    uint8_t* plane = (uint8_t*)(which ? c->vq : c->kq);
    uint16_t* sc = which ? c->vs : c->ks;
    const int type = plane_type(c->type, which);
    uint8_t* qrow = plane + row * kv_row_bytes(type, c->D);
    if (type == ORC_KV_F32) {
        float* f = (float*)qrow;
        for (int d = 0; d < c->D; ++d) f[d] = (float)orc_bf16_to_double(src[d]);
        return;
    }
    float* x = malloc((size_t)c->D * sizeof(float));
    for (int d = 0; d < c->D; ++d) x[d] = (float)orc_bf16_to_double(src[d]);
    if (kv_rotated(c->type)) orc_fwht_f32(c->D, x);   /* keys and values alike */
    uint16_t* srow = sc + row * (c->D / 32);
    for (int blk = 0; blk < c->D / 32; ++blk) {
        if (type == ORC_KV_Q8_0)
            orc_quantize_q8_0(x + 32 * blk, (int8_t*)qrow + 32 * blk, &srow[blk]);
        else if (type == ORC_KV_TQ3_0)
            orc_quantize_tq3_0(x + 32 * blk, qrow + 12 * blk, &srow[blk]);
        else
            orc_quantize_q4_0(x + 32 * blk, qrow + 16 * blk, &srow[blk]);
    }
    free(x);
}

static int attn_dims_ok(int B, int N, int Hq, int Hkv, int D, int cap, int window, int type) {
    if (B < 1 || N < 1 || N > 64 || Hkv < 1 || Hq < Hkv || Hq % Hkv != 0) return 0;
    if (D < 1 || cap < 1 || window < 0) return 0;
    if (type < ORC_KV_Q8_0 || type > ORC_KV_TQ3_0) return 0;
    if (type != ORC_KV_F32 && D % 32 != 0) return 0;
    if (kv_rotated(type) && (D & (D - 1)) != 0) return 0;   /* the rotation needs a power of two */
    return 1;
}

/* Visibility of a key at absolute position jpos to a node at position ipos:
 * causal (jpos <= ipos, guaranteed by the callers) and, with a window W > 0,
 * at most W positions back including the node itself. */
static int in_window(int jpos, int ipos, int window) {
    return window == 0 || jpos > ipos - window;
}

/* One output row: node i of sequence b, query head h, attending to every
 * visible key -- the cached positions j < P inside the window and the tree
 * slots of i's ancestors-or-self -- with an fp64 max-subtracted softmax. */
static void attn_one(const kv_cache* c, int N, int Hq, int window, double scale,
                     int b, int i, int h, int P, int n, const int32_t* depth,
                     const uint64_t* anc, const uint16_t* q, double* qd, double* key,
                     double* val, double* acc, float* out) {
    int D = c->D;
    int kvh = h / (Hq / c->Hkv);
    int ipos = P + depth[i];
    const uint16_t* qrow = q + (((size_t)b * N + i) * Hq + h) * D;
    for (int d = 0; d < D; ++d) qd[d] = orc_bf16_to_double(qrow[d]);
    if (kv_rotated(c->type)) fwht_f64(D, qd);   /* the query into the keys' basis */
    /* pass 1: the maximum score */
    double mx = -INFINITY;
    for (int slot = 0; slot < P + n; ++slot) {
        int jpos;
        if (slot < P) jpos = slot;
        else {
            int l = slot - P;
            if (!((anc[i] >> l) & 1ull)) continue;
            jpos = P + depth[l];
        }
        if (!in_window(jpos, ipos, window)) continue;
        kv_read_row(c, 0, b, kvh, slot, key);
        double s = 0.0;
        for (int d = 0; d < D; ++d) s += qd[d] * key[d];
        s *= scale;
        if (s > mx) mx = s;
    }
    /* pass 2: softmax-weighted sum of the values */
    double den = 0.0;
    for (int d = 0; d < D; ++d) acc[d] = 0.0;
    for (int slot = 0; slot < P + n; ++slot) {
        int jpos;
        if (slot < P) jpos = slot;
        else {
            int l = slot - P;
            if (!((anc[i] >> l) & 1ull)) continue;
            jpos = P + depth[l];
        }
        if (!in_window(jpos, ipos, window)) continue;
        kv_read_row(c, 0, b, kvh, slot, key);
        double s = 0.0;
        for (int d = 0; d < D; ++d) s += qd[d] * key[d];
        s *= scale;
        double p = exp(s - mx);
        den += p;
        kv_read_row(c, 1, b, kvh, slot, val);
        for (int d = 0; d < D; ++d) acc[d] += p * val[d];
    }
    float* o = out + (((size_t)b * N + i) * Hq + h) * D;
    for (int d = 0; d < D; ++d) acc[d] /= den;
    if (kv_rotated(c->type)) fwht_f64(D, acc);  /* back from the values' basis */
    for (int d = 0; d < D; ++d) o[d] = (float)acc[d];
}

int orc_tree_attn_verify(int B, int N, int Hq, int Hkv, int D, int cap, int window,
                         int kv_type, double scale,
                         const int32_t* parent, const int32_t* n_nodes, const int32_t* n_past,
                         const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                         void* kq, void* vq, uint16_t* ks, uint16_t* vs, float* out,
                         const int32_t* rows, int n_rows) {
    if (!attn_dims_ok(B, N, Hq, Hkv, D, cap, window, kv_type)) return ORC_ERR_ARG;
    kv_cache c = {B, Hkv, D, cap, kv_type, kq, vq, ks, vs};
    int32_t* depth = malloc((size_t)B * 64 * sizeof(int32_t));
    uint64_t* anc = malloc((size_t)B * 64 * sizeof(uint64_t));
    int rc = ORC_OK;
    for (int b = 0; b < B && rc == ORC_OK; ++b) {
        int n = n_nodes[b], P = n_past[b];
        if (n > N || orc_tree_topology(n, parent + (size_t)b * N, depth + 64 * b, anc + 64 * b) != ORC_OK)
            rc = ORC_ERR_TOPOLOGY;
        else if (P < 0 || P + n > cap)
            rc = ORC_ERR_CAPACITY;
    }
    /* (i) the tree's keys and values go into slots P .. P+n-1 first, so the
     * tree attends to exactly what a sequential decode would have stored. */
    for (int b = 0; b < B && rc == ORC_OK; ++b)
        for (int i = 0; i < n_nodes[b]; ++i)
            for (int h = 0; h < Hkv; ++h) {
                size_t off = (((size_t)b * N + i) * Hkv + h) * D;
                kv_write_row(&c, 0, b, h, n_past[b] + i, k_new + off);
                kv_write_row(&c, 1, b, h, n_past[b] + i, v_new + off);
            }
    /* (ii) every requested (sequence, node, query head) output; the rows
     * are independent, whichever thread computes them */
    if (rc == ORC_OK) {
        long n_out = 0;
        if (rows == NULL) {
            for (int b = 0; b < B; ++b) n_out += (long)n_nodes[b] * Hq;
        } else {
            for (int r = 0; r < n_rows; ++r) {
                int i = (rows[r] / Hq) % N, b = rows[r] / Hq / N;
                if (b < 0 || b >= B || i >= n_nodes[b]) rc = ORC_ERR_ARG;
            }
            n_out = n_rows;
        }
        if (rc == ORC_OK) {
#pragma omp parallel
            {
                double* qd = malloc(D * sizeof(double));
                double* key = malloc(D * sizeof(double));
                double* val = malloc(D * sizeof(double));
                double* acc = malloc(D * sizeof(double));
#pragma omp for schedule(dynamic)
                for (long r = 0; r < n_out; ++r) {
                    int b, i, h;
                    if (rows == NULL) {
                        long t = r;
                        b = 0;
                        while (t >= (long)n_nodes[b] * Hq) t -= (long)n_nodes[b++] * Hq;
                        i = (int)(t / Hq);
                        h = (int)(t % Hq);
                    } else {
                        h = rows[r] % Hq;
                        i = (rows[r] / Hq) % N;
                        b = rows[r] / Hq / N;
                    }
                    attn_one(&c, N, Hq, window, scale, b, i, h, n_past[b], n_nodes[b],
                             depth + 64 * b, anc + 64 * b, q, qd, key, val, acc, out);
                }
                free(qd); free(key); free(val); free(acc);
            }
        }
    }
    free(depth); free(anc);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* greedy acceptance                                                         */
/* ------------------------------------------------------------------------ */

int orc_accept_greedy(int B, int N, int V, const float* logits, const int32_t* tokens,
                      const int32_t* parent, const int32_t* n_nodes,
                      int32_t* path, int32_t* path_len, int32_t* next_token, int32_t* best) {
    if (B < 1 || N < 1 || N > 64 || V < 1) return ORC_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        int n = n_nodes[b];
        int32_t depth[64];
        uint64_t anc[64];
        const int32_t* par = parent + (size_t)b * N;
        if (n > N || orc_tree_topology(n, par, depth, anc) != ORC_OK) return ORC_ERR_TOPOLOGY;
        /* target argmax of every node; ties go to the lowest vocab index, and
         * a NaN logit counts as -infinity (an all-NaN row gives index 0) */
        for (int i = 0; i < n; ++i) {
            const float* row = logits + ((size_t)b * N + i) * V;
            int arg = 0;
            float top = isnan(row[0]) ? -INFINITY : row[0];
            for (int t = 1; t < V; ++t) {
                const float x = isnan(row[t]) ? -INFINITY : row[t];
                if (x > top) {
                    top = x;
                    arg = t;
                }
            }
            best[(size_t)b * N + i] = arg;
        }
        /* walk from the root while a child carries the target's argmax token;
         * among several matching children the lowest node index wins */
        int cur = 0, L = 0;
        path[(size_t)b * N + L++] = 0;
        for (;;) {
            int nxt = -1;
            for (int c = cur + 1; c < n; ++c)
                if (par[c] == cur && tokens[(size_t)b * N + c] == best[(size_t)b * N + cur]) {
                    nxt = c;
                    break;
                }
            if (nxt < 0) break;
            path[(size_t)b * N + L++] = nxt;
            cur = nxt;
        }
        path_len[b] = L;
        next_token[b] = best[(size_t)b * N + cur];
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* KV commit                                                                 */
/* ------------------------------------------------------------------------ */

int orc_kv_commit(int B, int N, int Hkv, int D, int cap, int kv_type,
                  const int32_t* path, const int32_t* path_len, const int32_t* n_past,
                  void* kq, void* vq, uint16_t* ks, uint16_t* vs) {
    /* The accepted nodes' keys and values move to the slots a sequential
     * decode would have used: slot P + path[m] -> slot P + m, m < L.  All
     * source rows are read before any is written, because a destination can
     * be another accepted node's source (path [0, 2, 3]: 2 -> 1, 3 -> 2). */
    if (B < 1 || N < 1 || N > 64 || Hkv < 1 || D < 1 || cap < 1) return ORC_ERR_ARG;
    if (kv_type < ORC_KV_Q8_0 || kv_type > ORC_KV_TQ3_0) return ORC_ERR_ARG;
    kv_cache c = {B, Hkv, D, cap, kv_type, kq, vq, ks, vs};
    size_t sb = (kv_type == ORC_KV_F32) ? 0 : (size_t)(D / 32) * sizeof(uint16_t);
    uint8_t* tmp = malloc((size_t)N * ((size_t)D * 4 + sb));
    for (int b = 0; b < B; ++b) {
        int L = path_len[b], P = n_past[b];
        if (L < 1 || L > N) { free(tmp); return ORC_ERR_ARG; }
        for (int m = 0; m < L; ++m) {
            int src = path[(size_t)b * N + m];
            if (src < 0 || src >= N || P + src >= cap || P < 0) { free(tmp); return ORC_ERR_CAPACITY; }
        }
        for (int h = 0; h < Hkv; ++h)
            for (int which = 0; which < 2; ++which) {
                const size_t qb = kv_row_bytes(plane_type(kv_type, which), D);
                uint8_t* plane = (uint8_t*)(which ? c.vq : c.kq);
                uint8_t* sc = (uint8_t*)(which ? c.vs : c.ks);
                for (int m = 0; m < L; ++m) {
                    size_t row = kv_row_index(&c, b, h, P + path[(size_t)b * N + m]);
                    memcpy(tmp + (size_t)m * (qb + sb), plane + row * qb, qb);
                    if (sb) memcpy(tmp + (size_t)m * (qb + sb) + qb, sc + row * sb, sb);
                }
                for (int m = 0; m < L; ++m) {
                    size_t row = kv_row_index(&c, b, h, P + m);
                    memcpy(plane + row * qb, tmp + (size_t)m * (qb + sb), qb);
                    if (sb) memcpy(sc + row * sb, tmp + (size_t)m * (qb + sb) + qb, sb);
                }
            }
    }
    free(tmp);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* tree-aware short convolution                                              */
/* ------------------------------------------------------------------------ */

int orc_tree_conv_verify(int B, int N, int C, int K, const int32_t* parent, const int32_t* n_nodes,
                         const uint16_t* x, const uint16_t* state, const float* w, float* out) {
    if (B < 1 || N < 1 || N > 64 || C < 1 || K < 2) return ORC_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        int n = n_nodes[b];
        int32_t depth[64];
        uint64_t anc[64];
        if (n < 1 || n > N) return ORC_ERR_TOPOLOGY;
        int rc = orc_tree_topology(n, parent + (size_t)b * N, depth, anc);
        if (rc != ORC_OK) return rc;
        for (int i = 0; i < n; ++i)
            for (int c = 0; c < C; ++c) {
                double acc = 0.0;
                /* walk back from node i: window position j = K-1, K-2, ... */
                int node = i, before_root = 0;
                for (int j = K - 1; j >= 0; --j) {
                    double v;
                    if (node >= 0) {
                        v = orc_bf16_to_double(x[((size_t)b * N + node) * C + c]);
                        node = parent[(size_t)b * N + node];
                    } else {
                        /* the (before_root+1)-th input before the root */
                        v = orc_bf16_to_double(state[((size_t)b * (K - 1) + (K - 2 - before_root)) * C + c]);
                        ++before_root;
                    }
                    acc += (double)w[(size_t)c * K + j] * v;
                }
                out[((size_t)b * N + i) * C + c] = (float)acc;
            }
    }
    return ORC_OK;
}

int orc_conv_commit(int B, int N, int C, int K, const uint16_t* x, const int32_t* path,
                    const int32_t* path_len, uint16_t* state) {
    if (B < 1 || N < 1 || C < 1 || K < 2) return ORC_ERR_ARG;
    uint16_t* seq = malloc((size_t)(K - 1 + N) * sizeof(uint16_t));
    for (int b = 0; b < B; ++b) {
        int L = path_len[b];
        if (L < 0 || L > N) { free(seq); return ORC_ERR_ARG; }
        for (int m = 0; m < L; ++m) {
            int p = path[(size_t)b * N + m];
            if (p < 0 || p >= N) { free(seq); return ORC_ERR_ARG; }
        }
        for (int c = 0; c < C; ++c) {
            /* the sequence [state ; x of the path], then its last K-1 entries */
            for (int t = 0; t < K - 1; ++t) seq[t] = state[((size_t)b * (K - 1) + t) * C + c];
            for (int m = 0; m < L; ++m) seq[K - 1 + m] = x[((size_t)b * N + path[(size_t)b * N + m]) * C + c];
            for (int t = 0; t < K - 1; ++t) state[((size_t)b * (K - 1) + t) * C + c] = seq[L + t];
        }
    }
    free(seq);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* threads                                                                   */
/* ------------------------------------------------------------------------ */

int orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}
