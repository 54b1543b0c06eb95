/*
 * msda_oracle.c -- fp64 CPU oracle for the multi-scale deformable attention
 * sampling core.  TEST INFRASTRUCTURE ONLY: it is called by the tests, by the
 * smoke check and by the benchmark's CPU-baseline leg, never by the product
 * path.  It shares no code with the CUDA library.
 *
 * What it computes (msda-triton README, "The operator"; course ch. 4,
 * "Bilinear sampling" and "Accumulate and store"; course ch. 5, "What the
 * backward pass must produce"):
 *
 *   out[b,q,m,:] = sum_l sum_k A[b,q,m,l,k] * bilinear_l(b, m, x_im, y_im)
 *   x_im = x * W_l - 0.5,  y_im = y * H_l - 0.5        (align_corners=False)
 *   x0 = floor(x_im), y0 = floor(y_im), lx = x_im - x0, ly = y_im - y0
 *   corner (y0+i, x0+j), i,j in {0,1}, weight w_ij = (i ? ly : 1-ly) * (j ? lx : 1-lx)
 *   a corner outside [0,W_l) x [0,H_l) contributes nothing (zero padding)
 *
 * and, with g = grad_out[b,q,m,:]:
 *
 *   grad_attn[p]     = sum_d g[d] * sampled[d]                 (output is linear in A)
 *   grad_loc[p][0]   = A * W_l * sum_d g[d] * d sampled[d] / d x_im
 *   grad_loc[p][1]   = A * H_l * sum_d g[d] * d sampled[d] / d y_im
 *   grad_value[b, start_l + (y0+i)*W_l + (x0+j), m, :] += A * w_ij * g   (valid corners)
 *
 * where the location derivative is that of the zero-padded bilinear
 * interpolant inside the cell [x0, x0+1] x [y0, y0+1] (the one-sided slope
 * implied by floor at integer coordinates).  Each sum above is taken over the
 * valid corners only, so a sample with no valid corner contributes nothing and
 * receives zero gradient.
 *
 * Coordinate precision.  The integer corner decision floor(x_im) is a
 * floating-point decision; the pages compute x_im in fp32.  coord_mode 1 does
 * the same (x_im = fp32 rounding of the exact x*W_l - 0.5, via one fused
 * multiply-add), so that the oracle and the kernel pick the same cell;
 * everything after the decision is fp64.  coord_mode 0 computes x_im exactly
 * in fp64 and is used for the mathematical checks (finite differences,
 * grid_sample restatement).
 *
 * Input dtypes (raw little-endian storage): 0 f32, 1 f16, 2 bf16, 3 f64.
 * Outputs are always fp64.  Index arithmetic is 64-bit throughout.
 * Parallelism: OpenMP over (b, m) pairs; each pair owns disjoint output rows
 * and a disjoint grad_value slice, so the summation order is fixed.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ODT_F32 = 0, ODT_F16 = 1, ODT_BF16 = 2, ODT_F64 = 3 };

/* ---- exact decoding of the storage formats (IEEE 754 binary16/32, bfloat16) ---- */

static double dec_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int man = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)man, -24);                 /* subnormal: man * 2^-24 */
    else if (e == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexp((double)(man + 1024), e - 25);     /* (1.man) * 2^(e-15) */
    return sign ? -v : v;
}

static double dec_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static double load_el(const void* base, int64_t i, int dt) {
    switch (dt) {
    case ODT_F32: return (double)((const float*)base)[i];
    case ODT_F16: return dec_f16(((const uint16_t*)base)[i]);
    case ODT_BF16: return dec_bf16(((const uint16_t*)base)[i]);
    default: return ((const double*)base)[i];
    }
}

/* ---- the shared problem description ---- */

typedef struct {
    int dt, coord_mode;      /* dt: value / grad_out storage */
    int64_t B, S, M, D, L, K, Q;
    const void* value;
    const int64_t* shapes;   /* [L,2] = (H, W) */
    const int64_t* starts;   /* [L] */
    const void* loc;         /* [B,Q,M,L,K,2] */
    const void* attn;        /* [B,Q,M,L,K] */
    int pdt;                 /* storage of loc / attn (dt unless a caller sets it) */
} prob_t;

/* One sampling point after the bilinear setup. */
typedef struct {
    double a;                /* attention weight */
    double lx, ly;           /* fractional offsets inside the cell */
    int64_t H, W;
    int valid[2][2];         /* [i][j]: corner (y0+i, x0+j) inside the level */
    int64_t row[2][2];       /* pyramid row index of each valid corner */
    double w[2][2];          /* bilinear weights */
    double dwdx[2][2];       /* d w_ij / d x_im */
    double dwdy[2][2];       /* d w_ij / d y_im */
} sample_t;

static void setup_sample(const prob_t* P, int64_t b, int64_t q, int64_t m, int64_t l, int64_t k,
                         sample_t* s) {
    int64_t p = (((b * P->Q + q) * P->M + m) * P->L + l) * P->K + k;
    double x = load_el(P->loc, 2 * p, P->pdt);
    double y = load_el(P->loc, 2 * p + 1, P->pdt);
    s->a = load_el(P->attn, p, P->pdt);
    s->H = P->shapes[2 * l];
    s->W = P->shapes[2 * l + 1];
    int64_t start = P->starts[l];

    double x_im, y_im;
    if (P->coord_mode == 1) {
        /* fp32 pixel coordinate: the exact x*W - 0.5 rounded once to binary32 */
        x_im = (double)fmaf((float)x, (float)s->W, -0.5f);
        y_im = (double)fmaf((float)y, (float)s->H, -0.5f);
    } else {
        x_im = x * (double)s->W - 0.5;
        y_im = y * (double)s->H - 0.5;
    }
    double x0 = floor(x_im), y0 = floor(y_im);
    s->lx = x_im - x0;
    s->ly = y_im - y0;

    for (int i = 0; i < 2; ++i) {
        for (int j = 0; j < 2; ++j) {
            double yy = y0 + i, xx = x0 + j;
            /* the comparisons are false for NaN / inf: such a corner is invalid */
            int ok = (xx >= 0.0) && (xx < (double)s->W) && (yy >= 0.0) && (yy < (double)s->H);
            s->valid[i][j] = ok;
            s->row[i][j] = ok ? start + (int64_t)yy * s->W + (int64_t)xx : -1;
            double wy = i ? s->ly : 1.0 - s->ly;
            double wx = j ? s->lx : 1.0 - s->lx;
            s->w[i][j] = wy * wx;
            s->dwdx[i][j] = wy * (j ? 1.0 : -1.0);
            s->dwdy[i][j] = wx * (i ? 1.0 : -1.0);
        }
    }
}

static inline int64_t value_index(const prob_t* P, int64_t b, int64_t row, int64_t m) {
    return ((b * P->S + row) * P->M + m) * P->D;
}

static int check_prob(const prob_t* P) {
    if (P->B < 0 || P->S < 0 || P->M < 0 || P->D < 0 || P->L < 0 || P->K < 0 || P->Q < 0) return -1;
    if (P->dt < 0 || P->dt > 3 || P->pdt < 0 || P->pdt > 3) return -2;
    for (int64_t l = 0; l < P->L; ++l) {
        int64_t H = P->shapes[2 * l], W = P->shapes[2 * l + 1], st = P->starts[l];
        if (H < 0 || W < 0 || st < 0 || st + H * W > P->S) return -3;
    }
    return 0;
}

/* ---- forward ---- */

/* out for one (b,q,m) unit into out[0..D) */
static void forward_unit(const prob_t* P, int64_t b, int64_t q, int64_t m, double* out) {
    for (int64_t d = 0; d < P->D; ++d) out[d] = 0.0;
    sample_t s;
    for (int64_t l = 0; l < P->L; ++l) {
        for (int64_t k = 0; k < P->K; ++k) {
            setup_sample(P, b, q, m, l, k, &s);
            for (int i = 0; i < 2; ++i)
                for (int j = 0; j < 2; ++j) {
                    if (!s.valid[i][j]) continue;
                    double c = s.a * s.w[i][j];
                    int64_t vi = value_index(P, b, s.row[i][j], m);
                    for (int64_t d = 0; d < P->D; ++d) out[d] += c * load_el(P->value, vi + d, P->dt);
                }
        }
    }
}

#define PROB_ARGS int dt, int coord_mode, int64_t B, int64_t S, int64_t M, int64_t D, int64_t L, \
    int64_t K, int64_t Q, const void* value, const int64_t* shapes, const int64_t* starts,      \
    const void* loc, const void* attn
/* dt: low byte = storage of value / grad_out; a non-zero high byte h gives
 * loc / attn the storage h - 1 (the fused oracle in oracle/__init__.py passes
 * the locations and weights it computes as fp64 arrays while value keeps the
 * I/O dtype); otherwise loc / attn share value's storage. */
#define PROB_INIT {dt & 0xff, coord_mode, B, S, M, D, L, K, Q, value, shapes, starts, loc, attn, \
                   (dt >> 8) ? ((dt >> 8) & 0xff) - 1 : (dt & 0xff)}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int msda_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* out: [B,Q,M,D] fp64 */
int msda_oracle_forward(PROB_ARGS, double* out, int nthreads) {
    prob_t P = PROB_INIT;
    int rc = check_prob(&P);
    if (rc) return rc;
    set_threads(nthreads);
    int64_t nbm = B * M;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bm = 0; bm < nbm; ++bm) {
        int64_t b = bm / M, m = bm % M;
        for (int64_t q = 0; q < Q; ++q) forward_unit(&P, b, q, m, out + ((b * Q + q) * M + m) * D);
    }
    return 0;
}

/* out for selected flat units u = (b*Q + q)*M + m; out: [n, D] */
int msda_oracle_forward_units(PROB_ARGS, const int64_t* units, int64_t n, double* out, int nthreads) {
    prob_t P = PROB_INIT;
    int rc = check_prob(&P);
    if (rc) return rc;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < n; ++i) {
        int64_t u = units[i];
        int64_t m = u % M, q = (u / M) % Q, b = u / (M * Q);
        forward_unit(&P, b, q, m, out + i * D);
    }
    return 0;
}

/* ---- backward ---- */

/* grad_loc[0..L*K*2) and grad_attn[0..L*K) of one unit; if gv != NULL also
 * scatter A*w_ij*g into the grad_value slice of (b, m). */
static void backward_unit(const prob_t* P, int64_t b, int64_t q, int64_t m, const void* grad_out,
                          double* gloc, double* gattn, double* gv) {
    const int64_t D = P->D;
    const int64_t gbase = ((b * P->Q + q) * P->M + m) * D;
    sample_t s;
    for (int64_t l = 0; l < P->L; ++l) {
        for (int64_t k = 0; k < P->K; ++k) {
            setup_sample(P, b, q, m, l, k, &s);
            double ga = 0.0, gx = 0.0, gy = 0.0;
            for (int i = 0; i < 2; ++i)
                for (int j = 0; j < 2; ++j) {
                    if (!s.valid[i][j]) continue;
                    int64_t vi = value_index(P, b, s.row[i][j], m);
                    double dot = 0.0;   /* <g, v_ij> */
                    for (int64_t d = 0; d < D; ++d)
                        dot += load_el(grad_out, gbase + d, P->dt) * load_el(P->value, vi + d, P->dt);
                    ga += s.w[i][j] * dot;
                    gx += s.dwdx[i][j] * dot;
                    gy += s.dwdy[i][j] * dot;
                    if (gv) {
                        double c = s.a * s.w[i][j];
                        for (int64_t d = 0; d < D; ++d) gv[vi + d] += c * load_el(grad_out, gbase + d, P->dt);
                    }
                }
            int64_t sl = l * P->K + k;
            gattn[sl] = ga;
            gloc[2 * sl] = s.a * (double)s.W * gx;
            gloc[2 * sl + 1] = s.a * (double)s.H * gy;
        }
    }
}

/* grad_value: [B,S,M,D] fp64 (overwritten); grad_loc: [B,Q,M,L,K,2]; grad_attn: [B,Q,M,L,K] */
int msda_oracle_backward(PROB_ARGS, const void* grad_out, double* grad_value, double* grad_loc,
                         double* grad_attn, int nthreads) {
    prob_t P = PROB_INIT;
    int rc = check_prob(&P);
    if (rc) return rc;
    set_threads(nthreads);
    int64_t nbm = B * M;
    const int64_t LK = L * K;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bm = 0; bm < nbm; ++bm) {
        int64_t b = bm / M, m = bm % M;
        /* zero this pair's grad_value slice */
        for (int64_t r = 0; r < S; ++r) {
            double* row = grad_value + value_index(&P, b, r, m);
            for (int64_t d = 0; d < D; ++d) row[d] = 0.0;
        }
        for (int64_t q = 0; q < Q; ++q) {
            int64_t u = (b * Q + q) * M + m;
            backward_unit(&P, b, q, m, grad_out, grad_loc + u * LK * 2, grad_attn + u * LK, grad_value);
        }
    }
    return 0;
}

/* grad_loc / grad_attn of selected units: gloc [n, L*K*2], gattn [n, L*K] */
int msda_oracle_backward_units(PROB_ARGS, const void* grad_out, const int64_t* units, int64_t n,
                               double* grad_loc, double* grad_attn, int nthreads) {
    prob_t P = PROB_INIT;
    int rc = check_prob(&P);
    if (rc) return rc;
    set_threads(nthreads);
    const int64_t LK = L * K;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < n; ++i) {
        int64_t u = units[i];
        int64_t m = u % M, q = (u / M) % Q, b = u / (M * Q);
        backward_unit(&P, b, q, m, grad_out, grad_loc + i * LK * 2, grad_attn + i * LK, NULL);
    }
    return 0;
}

/* grad_value of selected rows r = (b*S + pixel)*M + m, out: [n, D].
 * For each (b, m) that owns a requested row, every sample of that pair is
 * visited and the contributions of its valid corners to requested pixels are
 * summed in (q, l, k, corner) order. */
int msda_oracle_grad_value_rows(PROB_ARGS, const void* grad_out, const int64_t* rows, int64_t n,
                                double* out, int nthreads) {
    prob_t P = PROB_INIT;
    int rc = check_prob(&P);
    if (rc) return rc;
    set_threads(nthreads);
    for (int64_t i = 0; i < n * D; ++i) out[i] = 0.0;
    int64_t nbm = B * M;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bm = 0; bm < nbm; ++bm) {
        int64_t b = bm / M, m = bm % M;
        int64_t* slot = NULL;   /* pixel -> first requested row index, or -1 */
        for (int64_t i = 0; i < n; ++i) {
            int64_t r = rows[i];
            if (r % M != m || r / (M * S) != b) continue;
            if (!slot) {
                slot = (int64_t*)malloc(sizeof(int64_t) * (size_t)(S > 0 ? S : 1));
                for (int64_t t = 0; t < S; ++t) slot[t] = -1;
            }
            int64_t pix = (r / M) % S;
            if (slot[pix] < 0) slot[pix] = i;
        }
        if (!slot) continue;
        sample_t s;
        for (int64_t q = 0; q < Q; ++q) {
            int64_t gbase = ((b * Q + q) * M + m) * D;
            for (int64_t l = 0; l < L; ++l)
                for (int64_t k = 0; k < K; ++k) {
                    setup_sample(&P, b, q, m, l, k, &s);
                    for (int i = 0; i < 2; ++i)
                        for (int j = 0; j < 2; ++j) {
                            if (!s.valid[i][j]) continue;
                            int64_t t = slot[s.row[i][j]];
                            if (t < 0) continue;
                            double c = s.a * s.w[i][j];
                            for (int64_t d = 0; d < D; ++d)
                                out[t * D + d] += c * load_el(grad_out, gbase + d, P.dt);
                        }
                }
        }
        free(slot);
    }
    /* duplicate requests of the same row copy the first one's result */
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = 0; j < i; ++j)
            if (rows[j] == rows[i]) {
                memcpy(out + i * D, out + j * D, sizeof(double) * (size_t)D);
                break;
            }
    return 0;
}

/* ---- fused operator: sampling locations from reference points and offsets ----
 *
 * msda-triton README, "The operator": the sampling location is the reference
 * point mapped to level l plus the learned offset.  Reading taken: the
 * reference point [B,Q,L,2] is normalised to [0,1] and shared by all levels,
 * the offset [B,Q,M,L,K,2] is in pixels of level l, so
 *
 *   loc.x = ref.x + off.x / W_l,   loc.y = ref.y + off.y / H_l.
 *
 * coord_mode 1 takes each operation in binary32 with one rounding (the
 * quotient, then the sum), as the kernels do, so that the cell decision made
 * on the result matches theirs; coord_mode 0 takes them in fp64.  Inputs and
 * the output are fp64 (the inputs hold exactly representable binary32,
 * binary16 or bfloat16 values). */
int msda_oracle_fused_locations(int coord_mode, int64_t B, int64_t Q, int64_t M, int64_t L, int64_t K,
                                const int64_t* shapes, const double* ref, const double* off, double* loc) {
    if (B < 0 || Q < 0 || M < 0 || L < 1 || K < 1 || (coord_mode != 0 && coord_mode != 1)) return 1;
    for (int64_t l = 0; l < L; ++l)
        if (shapes[2 * l] < 1 || shapes[2 * l + 1] < 1) return 2;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t q = 0; q < Q; ++q)
            for (int64_t m = 0; m < M; ++m)
                for (int64_t l = 0; l < L; ++l) {
                    const double* r = ref + ((b * Q + q) * L + l) * 2;
                    double size[2] = {(double)shapes[2 * l + 1], (double)shapes[2 * l]};   /* (W, H) */
                    for (int64_t k = 0; k < K; ++k) {
                        int64_t p = (((b * Q + q) * M + m) * L + l) * K + k;
                        for (int c = 0; c < 2; ++c) {
                            double o = off[2 * p + c];
                            if (coord_mode == 1) {
                                float quot = (float)o / (float)size[c];
                                float sum = (float)r[c] + quot;
                                loc[2 * p + c] = (double)sum;
                            } else {
                                loc[2 * p + c] = r[c] + o / size[c];
                            }
                        }
                    }
                }
    return 0;
}
