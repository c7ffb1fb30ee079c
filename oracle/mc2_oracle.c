/*
 * mc2_oracle.c -- plain, slow, obviously-correct CPU oracle for the MC2
 * fused-linear hot path (AllGatherMatmul and AlltoAllQuantMatmul).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file.  Only the test suite, the smoke check of the entry module
 * and the CPU-baseline / reference arm of the benchmark use it.  It shares no
 * code, header, table or helper with the CUDA library: every conversion and
 * every formula below is written out again from the pages' definitions.
 *
 * Sources (page title -- section):
 *   [AG]  "torch_npu.npu_all_gather_base_mm" -- 功能说明 (function), 接口原型
 *         (prototype), 参数说明 (parameters), 输出说明 (outputs), 约束说明
 *         (constraints).
 *   [A2A] "aclnnAlltoAllQuantMatmul" -- 功能说明, 计算公式: 动态量化场景
 *         (dynamic-quant formula) and 全量化场景 (full-quant formula);
 *         约束说明 (constraints).
 *   [MC2] "hyper_parallel .../tensor_parallel/mc2.py" (coverage listing) --
 *         module docstring and AllGatherMatmulFunction.forward.
 *   [QAR] "QuantAllReduce" (ops-transformer mc2/quant_all_reduce) -- 功能说明
 *         (formula), 参数说明 (parameters), 约束说明 (constraints).
 *
 * Precision.  The pages do not fix the accumulation precision of the bf16 /
 * fp16 matmul, so the oracle accumulates in fp64 and rounds once to the
 * output type.  Every step that decides an integer (the int8 quantised value)
 * or that the pages order explicitly (the dequant products) is done in fp32,
 * the precision the kernel uses, one IEEE operation at a time.  Build with
 * -ffp-contract=off so that no multiply-add is fused.
 *
 * Where a function has no independent pin it says so; every function below
 * is pinned by the not-gpu tests (closed forms, brute force, invariants).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_ERR_ARG -1
#define OR_ERR_OVERFLOW -2
#define OR_ERR_NOMEM -3

/* ------------------------------------------------------------------------ */
/* 16-bit floating formats, from the IEEE-754 binary16 and bfloat16 layouts. */
/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits.                 */
/* binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits.                 */
/* ------------------------------------------------------------------------ */

static void fmt_params(int is_bf16, int *frac_bits, int *exp_bits, int *bias) {
    *frac_bits = is_bf16 ? 7 : 10;
    *exp_bits = is_bf16 ? 8 : 5;
    *bias = (1 << (*exp_bits - 1)) - 1;
}

/* Exact value of a 16-bit encoding as a double. */
double oracle_decode16(uint16_t v, int is_bf16) {
    int fb, eb, bias;
    fmt_params(is_bf16, &fb, &eb, &bias);
    int sign = (v >> 15) & 1;
    int e = (v >> fb) & ((1 << eb) - 1);
    int f = v & ((1 << fb) - 1);
    double r;
    if (e == (1 << eb) - 1)
        r = f ? NAN : INFINITY;
    else if (e == 0)
        r = ldexp((double)f, 1 - bias - fb);               /* subnormal */
    else
        r = ldexp((double)(f | (1 << fb)), e - bias - fb); /* normal */
    return sign ? -r : r;
}

/* Round a double to the nearest 16-bit value, ties to even, directly (one
 * rounding, no detour through fp32).  Overflow gives infinity. */
uint16_t oracle_encode16_rne(double x, int is_bf16) {
    int fb, eb, bias;
    fmt_params(is_bf16, &fb, &eb, &bias);
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    uint16_t inf = (uint16_t)(((1u << eb) - 1u) << fb);
    if (isnan(x)) return (uint16_t)(sign | inf | (1u << (fb - 1)));
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | inf);
    int e2;
    (void)frexp(a, &e2);          /* a = g * 2^e2, g in [0.5, 1) */
    int E = e2 - 1;               /* exponent of the leading bit */
    int emin = 1 - bias;
    if (E < emin) E = emin;       /* subnormal range: fixed quantum */
    /* quantum = 2^(E - fb); scale a to units of the quantum (exact) */
    double s = ldexp(a, fb - E);
    double r = nearbyint(s);      /* default mode: nearest, ties to even */
    uint32_t ri = (uint32_t)r;
    if (ri == (1u << (fb + 1))) { /* rounded up into the next binade */
        ri >>= 1;
        E += 1;
    }
    uint32_t efield, ffield;
    if (ri < (1u << fb)) {        /* subnormal (only when E == emin) */
        efield = 0;
        ffield = ri;
    } else {
        efield = (uint32_t)(E + bias);
        ffield = ri - (1u << fb);
    }
    if (efield >= (1u << eb) - 1u) return (uint16_t)(sign | inf);
    return (uint16_t)(sign | (efield << fb) | ffield);
}

/* Bulk helpers (used by the Python wrapper and the pins). */
void oracle_decode16_array(const uint16_t *in, int64_t count, int is_bf16, double *out) {
    for (int64_t i = 0; i < count; ++i) out[i] = oracle_decode16(in[i], is_bf16);
}

void oracle_encode16_array(const double *in, int64_t count, int is_bf16, uint16_t *out) {
    for (int64_t i = 0; i < count; ++i) out[i] = oracle_encode16_rne(in[i], is_bf16);
}

/* All 65536 decodings as fp32 (every 16-bit value is exact in fp32). */
static void build_decode_table(int is_bf16, float *table) {
    for (uint32_t v = 0; v < 65536u; ++v) table[v] = (float)oracle_decode16((uint16_t)v, is_bf16);
}

/* ------------------------------------------------------------------------ */
/* [AG] AllGatherMatmul.                                                     */
/*   gathered = AllGather_m(input)  -- the second output (输出说明)          */
/*   out      = gathered @ x2 (+ bias)  -- the first output                  */
/* Row i of the gathered matrix is row (i mod m_local) of rank (i div        */
/* m_local)'s shard: AllGather concatenates the world_size shards along m.   */
/* x2 is (k, n) row-major, or, with x2_is_nk, the nn.Linear weight w (n, k)  */
/* with x2 = w^T ([AG] 约束说明: x2 may be passed transposed; [MC2]          */
/* AllGatherMatmulFunction.forward passes w.t()).                            */
/* bias (n) is added before the single rounding to the output type ([AG]     */
/* 参数说明 bias is 1-D of size n; [MC2] forward adds it after the op).      */
/* ------------------------------------------------------------------------ */

/* Explicit copy-concat of the shards along m. */
int oracle_gather(const uint16_t *const *chunks, int world_size, int64_t m_local, int64_t k,
                  uint16_t *gathered) {
    if (!chunks || !gathered || world_size < 1 || m_local < 0 || k < 0) return OR_ERR_ARG;
    for (int r = 0; r < world_size; ++r)
        memcpy(gathered + (int64_t)r * m_local * k, chunks[r], (size_t)(m_local * k) * sizeof(uint16_t));
    return OR_OK;
}

/* out[ii, j] for each requested gathered row i = rows[ii] (all rows when rows is NULL). */
int oracle_all_gather_mm(const uint16_t *const *chunks, int world_size, int64_t m_local, int64_t k,
                         const uint16_t *x2, int64_t n, int x2_is_nk, const uint16_t *bias,
                         int is_bf16, const int64_t *rows, int64_t n_rows, uint16_t *out) {
    if (!chunks || !x2 || !out || world_size < 1 || m_local < 1 || k < 1 || n < 1) return OR_ERR_ARG;
    int64_t m = (int64_t)world_size * m_local;
    if (!rows) n_rows = m;
    for (int64_t ii = 0; ii < n_rows; ++ii) {
        int64_t i = rows ? rows[ii] : ii;
        if (i < 0 || i >= m) return OR_ERR_ARG;
    }
    float *tab = (float *)malloc(65536 * sizeof(float));
    if (!tab) return OR_ERR_NOMEM;
    build_decode_table(is_bf16, tab);
    int err = OR_OK;
#pragma omp parallel
    {
        double *acc = (double *)malloc((size_t)n * sizeof(double));
        if (!acc) {
#pragma omp atomic write
            err = OR_ERR_NOMEM;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t ii = 0; ii < n_rows; ++ii) {
                int64_t i = rows ? rows[ii] : ii;
                int64_t r = i / m_local;          /* which rank's shard */
                int64_t li = i - r * m_local;     /* row inside that shard */
                const uint16_t *arow = chunks[r] + li * k;
                for (int64_t j = 0; j < n; ++j) acc[j] = 0.0;
                if (!x2_is_nk) {
                    /* acc[j] = sum over ascending kk of A[i,kk] * x2[kk,j] */
                    for (int64_t kk = 0; kk < k; ++kk) {
                        double a = tab[arow[kk]];
                        const uint16_t *brow = x2 + kk * n;
                        for (int64_t j = 0; j < n; ++j) acc[j] += a * (double)tab[brow[j]];
                    }
                } else {
                    /* x2[kk,j] = w[j,kk] */
                    for (int64_t j = 0; j < n; ++j) {
                        const uint16_t *wrow = x2 + j * k;
                        double s = 0.0;
                        for (int64_t kk = 0; kk < k; ++kk) s += (double)tab[arow[kk]] * (double)tab[wrow[kk]];
                        acc[j] = s;
                    }
                }
                for (int64_t j = 0; j < n; ++j) {
                    double v = acc[j] + (bias ? (double)tab[bias[j]] : 0.0);
                    out[ii * n + j] = oracle_encode16_rne(v, is_bf16);
                }
            }
            free(acc);
        }
    }
    free(tab);
    return err;
}

/* ------------------------------------------------------------------------ */
/* [A2A] AlltoAllQuantMatmul.                                                */
/*   commOut      = AlltoAll(x1.view(rankSize, BS/rankSize, H))              */
/*   permutedOut  = commOut.permute(1, 0, 2).view(BS/rankSize, rankSize*H)   */
/* The rank's received blocks are commOut[r] = chunk r, each (BS/R, H).      */
/* permute(1,0,2) then view gives permutedOut[t, r*H + h] = chunk_r[t, h].   */
/* [A2A] commOut = AlltoAll(x1.view(rankSize, BS/rankSize, H)): after the
 * exchange, block r of this rank's commOut (rankSize, BS/rankSize, H) is what
 * rank r sent it, i.e. received chunk r.  commOut[r, t, hh] = chunk_r[t, hh],
 * returned as the optional alltoAllOut output (same dtype as x1). */
int oracle_comm_out(const void *const *chunks, int rank_size, int64_t bs_local, int64_t h, int elem_bytes,
                    void *comm_out) {
    if (!chunks || !comm_out || rank_size < 1 || bs_local < 1 || h < 1) return OR_ERR_ARG;
    if (elem_bytes != 1 && elem_bytes != 2) return OR_ERR_ARG;
    for (int r = 0; r < rank_size; ++r) {
        for (int64_t t = 0; t < bs_local; ++t) {
            for (int64_t hh = 0; hh < h; ++hh) {
                int64_t dst = ((int64_t)r * bs_local + t) * h + hh;
                int64_t src = t * h + hh;
                if (elem_bytes == 1)
                    ((int8_t *)comm_out)[dst] = ((const int8_t *)chunks[r])[src];
                else
                    ((uint16_t *)comm_out)[dst] = ((const uint16_t *)chunks[r])[src];
            }
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */

int oracle_permute(const void *const *chunks, int rank_size, int64_t bs_local, int64_t h,
                   int elem_bytes, const int64_t *rows, int64_t n_rows, void *permuted) {
    if (!chunks || !permuted || rank_size < 1 || bs_local < 1 || h < 1) return OR_ERR_ARG;
    if (elem_bytes != 1 && elem_bytes != 2) return OR_ERR_ARG;
    if (!rows) n_rows = bs_local;
    int64_t cols = (int64_t)rank_size * h;
    for (int64_t ii = 0; ii < n_rows; ++ii) {
        int64_t t = rows ? rows[ii] : ii;
        if (t < 0 || t >= bs_local) return OR_ERR_ARG;
        for (int r = 0; r < rank_size; ++r) {
            for (int64_t hh = 0; hh < h; ++hh) {
                int64_t dst = ii * cols + (int64_t)r * h + hh;
                int64_t src = t * h + hh;
                if (elem_bytes == 1)
                    ((int8_t *)permuted)[dst] = ((const int8_t *)chunks[r])[src];
                else
                    ((uint16_t *)permuted)[dst] = ((const uint16_t *)chunks[r])[src];
            }
        }
    }
    return OR_OK;
}

/* [A2A] 动态量化场景:  permutedOut_quant, x1_scale = Quant(permutedOut * x1ScaleOptional)
 * Per-token (one scale per row, quant mode 7 "pertoken动态量化") symmetric
 * int8.  Readings where the page is silent: y = P * s in fp32 (exact for
 * 16-bit inputs); scale = max|y| / 127 (IEEE fp32 division); q = y / scale
 * (IEEE fp32 division) rounded to nearest, ties to even, clamped to
 * [-127, 127]; an all-zero row gets scale 0 and q 0; a missing smooth scale
 * means s = 1. */
int oracle_quant_pertoken_dynamic(const uint16_t *permuted, int64_t n_rows, int64_t cols,
                                  const uint16_t *smooth, int is_bf16, int8_t *q, float *x1_scale) {
    if (!permuted || !q || !x1_scale || n_rows < 0 || cols < 1) return OR_ERR_ARG;
    for (int64_t t = 0; t < n_rows; ++t) {
        const uint16_t *row = permuted + t * cols;
        float amax = 0.0f;
        for (int64_t c = 0; c < cols; ++c) {
            float x = (float)oracle_decode16(row[c], is_bf16);
            float s = smooth ? (float)oracle_decode16(smooth[c], is_bf16) : 1.0f;
            float y = x * s;
            float ay = fabsf(y);
            if (ay > amax) amax = ay;
        }
        float scale = amax / 127.0f;
        x1_scale[t] = scale;
        for (int64_t c = 0; c < cols; ++c) {
            int8_t qv = 0;
            if (scale != 0.0f) {
                float x = (float)oracle_decode16(row[c], is_bf16);
                float s = smooth ? (float)oracle_decode16(smooth[c], is_bf16) : 1.0f;
                float y = x * s;
                float v = y / scale;
                float rv = nearbyintf(v);
                if (rv > 127.0f) rv = 127.0f;
                if (rv < -127.0f) rv = -127.0f;
                qv = (int8_t)rv;
            }
            q[t * cols + c] = qv;
        }
    }
    return OR_OK;
}

/* [A2A] output_quant = permutedOut_quant @ x2: int8 x int8 summed exactly.
 * Accumulates in int64 and fails if a result does not fit in int32. */
int oracle_int8_mm(const int8_t *a, int64_t n_rows, int64_t k, const int8_t *x2, int64_t n, int32_t *acc) {
    if (!a || !x2 || !acc || n_rows < 0 || k < 1 || n < 1) return OR_ERR_ARG;
    int err = OR_OK;
#pragma omp parallel
    {
        int64_t *s = (int64_t *)malloc((size_t)n * sizeof(int64_t));
        if (!s) {
#pragma omp atomic write
            err = OR_ERR_NOMEM;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t t = 0; t < n_rows; ++t) {
                for (int64_t j = 0; j < n; ++j) s[j] = 0;
                for (int64_t kk = 0; kk < k; ++kk) {
                    int64_t av = a[t * k + kk];
                    const int8_t *brow = x2 + kk * n;
                    for (int64_t j = 0; j < n; ++j) s[j] += av * (int64_t)brow[j];
                }
                for (int64_t j = 0; j < n; ++j) {
                    if (s[j] > INT32_MAX || s[j] < INT32_MIN) {
#pragma omp atomic write
                        err = OR_ERR_OVERFLOW;
                    }
                    acc[t * n + j] = (int32_t)s[j];
                }
            }
            free(s);
        }
    }
    return err;
}

/* [A2A] output = output_quant x x1_scale x x2_scale; output = output + bias.
 * fp32, one IEEE operation at a time, left to right as the formula prints
 * it: ((float(acc) * x1_scale[t]) * x2_scale[j]) + bias[j], then one
 * rounding to bfloat16 (ties to even).  x2_scale is per channel (quant mode
 * 2 "perchannel"). */
int oracle_dequant(const int32_t *acc, int64_t n_rows, int64_t n, const float *x1_scale,
                   const float *x2_scale, const float *bias, uint16_t *out_bf16) {
    if (!acc || !x1_scale || !x2_scale || !out_bf16 || n_rows < 0 || n < 1) return OR_ERR_ARG;
    for (int64_t t = 0; t < n_rows; ++t) {
        for (int64_t j = 0; j < n; ++j) {
            float v = (float)acc[t * n + j];
            v = v * x1_scale[t];
            v = v * x2_scale[j];
            if (bias) v = v + bias[j];
            out_bf16[t * n + j] = oracle_encode16_rne((double)v, 1);
        }
    }
    return OR_OK;
}

/* The whole AlltoAllQuantMatmul path for the requested permuted rows.
 *   quant_mode 7 (dynamic): chunks are 16-bit (is_bf16 selects bf16/fp16),
 *     x1_scale_in is the optional smooth scale (rank_size*h, same type).
 *   quant_mode 3 (full quant, pertoken): chunks are int8, x1_scale_in is the
 *     per-token fp32 scale (bs_local).  The page prints x1 @ x2 in this
 *     scenario; the permuted matrix is the only operand whose shape matches
 *     x2, so it is read as permutedOut @ x2.
 * Optional outputs: q_out (n_rows, rank_size*h), x1_scale_out (n_rows),
 * acc_out (n_rows, n). */
int oracle_alltoall_quant_mm(const void *const *chunks, int rank_size, int64_t bs_local, int64_t h,
                             int quant_mode, int is_bf16, const void *x1_scale_in, const int8_t *x2,
                             const float *x2_scale, const float *bias, int64_t n, const int64_t *rows,
                             int64_t n_rows, uint16_t *out, int8_t *q_out, float *x1_scale_out,
                             int32_t *acc_out) {
    if (!chunks || !x2 || !x2_scale || !out || rank_size < 1 || bs_local < 1 || h < 1 || n < 1)
        return OR_ERR_ARG;
    if (quant_mode != 3 && quant_mode != 7) return OR_ERR_ARG;
    if (quant_mode == 3 && !x1_scale_in) return OR_ERR_ARG;
    if (!rows) n_rows = bs_local;
    int64_t cols = (int64_t)rank_size * h;
    int err = OR_OK;
    int8_t *q = (int8_t *)malloc((size_t)(n_rows * cols));
    float *sc = (float *)malloc((size_t)n_rows * sizeof(float));
    int32_t *acc = (int32_t *)malloc((size_t)(n_rows * n) * sizeof(int32_t));
    void *perm = malloc((size_t)(n_rows * cols) * (quant_mode == 7 ? 2 : 1));
    if (!q || !sc || !acc || !perm) {
        err = OR_ERR_NOMEM;
        goto done;
    }
    err = oracle_permute(chunks, rank_size, bs_local, h, quant_mode == 7 ? 2 : 1, rows, n_rows, perm);
    if (err) goto done;
    if (quant_mode == 7) {
        err = oracle_quant_pertoken_dynamic((const uint16_t *)perm, n_rows, cols,
                                            (const uint16_t *)x1_scale_in, is_bf16, q, sc);
        if (err) goto done;
    } else {
        memcpy(q, perm, (size_t)(n_rows * cols));
        for (int64_t ii = 0; ii < n_rows; ++ii) {
            int64_t t = rows ? rows[ii] : ii;
            sc[ii] = ((const float *)x1_scale_in)[t];
        }
    }
    err = oracle_int8_mm(q, n_rows, cols, x2, n, acc);
    if (err) goto done;
    err = oracle_dequant(acc, n_rows, n, sc, x2_scale, bias, out);
    if (err) goto done;
    if (q_out) memcpy(q_out, q, (size_t)(n_rows * cols));
    if (x1_scale_out) memcpy(x1_scale_out, sc, (size_t)n_rows * sizeof(float));
    if (acc_out) memcpy(acc_out, acc, (size_t)(n_rows * n) * sizeof(int32_t));
done:
    free(q);
    free(sc);
    free(acc);
    free(perm);
    return err;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* [MC2] MatmulReduceScatter ("hyper_parallel .../mc2.py", module docstring:  */
/*   matmul_reduce_scatter forward  Y = ReduceScatter_m(X @ W^T)), the dual    */
/* of AllGatherMatmul.  Rank r holds X_r (m, k_local) and its weight shard     */
/* W_r (n, k_local) (x2 = W_r^T, as MatmulReduceScatterFunction.forward        */
/* passes w.t()).  The rank partials P_r = X_r @ W_r^T (m, n) are summed and   */
/* the sum is scattered along m: rank j receives rows [j*m/R, (j+1)*m/R).     */
/* Reading: the sum is exact (fp64 here) and rounded once to the output type; */
/* bias (n), if given, is added before that rounding.                          */
/* out is the (m, n) concatenation of the R ranks' outputs (rank j = block j). */
/* ------------------------------------------------------------------------ */
int oracle_matmul_reduce_scatter(const uint16_t *const *x_chunks, const uint16_t *const *w_chunks, int world_size,
                                 int64_t m, int64_t k_local, int64_t n, int w_is_nk, const uint16_t *bias,
                                 int is_bf16, const int64_t *rows, int64_t n_rows, uint16_t *out) {
    if (!x_chunks || !w_chunks || !out || world_size < 1 || m < 1 || k_local < 1 || n < 1) return OR_ERR_ARG;
    if (!rows) n_rows = m;
    for (int64_t ii = 0; ii < n_rows; ++ii) {
        int64_t i = rows ? rows[ii] : ii;
        if (i < 0 || i >= m) return OR_ERR_ARG;
    }
    float *tab = (float *)malloc(65536 * sizeof(float));
    if (!tab) return OR_ERR_NOMEM;
    build_decode_table(is_bf16, tab);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t ii = 0; ii < n_rows; ++ii) {
        int64_t i = rows ? rows[ii] : ii;
        for (int64_t j = 0; j < n; ++j) {
            double s = 0.0;
            for (int r = 0; r < world_size; ++r) {        /* the reduction over ranks */
                const uint16_t *xrow = x_chunks[r] + i * k_local;
                for (int64_t kk = 0; kk < k_local; ++kk) {
                    /* W_r^T[kk, j] = W_r[j, kk] (w_is_nk) or x2_r[kk, j] */
                    uint16_t wv = w_is_nk ? w_chunks[r][j * k_local + kk] : w_chunks[r][kk * n + j];
                    s += (double)tab[xrow[kk]] * (double)tab[wv];
                }
            }
            if (bias) s += (double)tab[bias[j]];
            out[ii * n + j] = oracle_encode16_rne(s, is_bf16);
        }
    }
    free(tab);
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* [MC2] Weight and bias gradients of the fused linear layers                 */
/* ("hyper_parallel .../mc2.py": module docstring, dW = dY^T @ AllGather_m(X) */
/* for all_gather_matmul and dW = AllGather_m(dY)^T @ X for                    */
/* matmul_reduce_scatter; AllGatherMatmulFunction.backward: grad_w =          */
/* grad_out.t().matmul(gathered), grad_bias = grad_out.sum(dim=0)).            */
/*   dw[i, j] = sum_t dy[t, i] * x[t, j]     dy (m, n), x (m, k), dw (n, k)    */
/*   db[i]    = sum_t dy[t, i]                                   db (n)        */
/* Reading: both sums exact (fp64 here, ascending t) and rounded once to the   */
/* operand type.  dw is computed for the requested rows i (all when rows is    */
/* NULL) into dw (n_rows, k); db (all n) when db is non-NULL.                  */
/* ------------------------------------------------------------------------ */
int oracle_matmul_weight_grad(const uint16_t *dy, const uint16_t *x, int64_t m, int64_t n, int64_t k, int is_bf16,
                              const int64_t *rows, int64_t n_rows, uint16_t *dw, uint16_t *db) {
    if (!dy || !x || m < 1 || n < 1 || k < 1) return OR_ERR_ARG;
    if (!rows) n_rows = n;
    if (n_rows > 0 && !dw) return OR_ERR_ARG;
    for (int64_t ii = 0; ii < n_rows; ++ii) {
        int64_t i = rows ? rows[ii] : ii;
        if (i < 0 || i >= n) return OR_ERR_ARG;
    }
    float *tab = (float *)malloc(65536 * sizeof(float));
    if (!tab) return OR_ERR_NOMEM;
    build_decode_table(is_bf16, tab);
    int err = OR_OK;
#pragma omp parallel
    {
        double *acc = (double *)malloc((size_t)k * sizeof(double));
        if (!acc) {
#pragma omp atomic write
            err = OR_ERR_NOMEM;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t ii = 0; ii < n_rows; ++ii) {
            if (!acc) continue;
            int64_t i = rows ? rows[ii] : ii;
            for (int64_t j = 0; j < k; ++j) acc[j] = 0.0;
            for (int64_t t = 0; t < m; ++t) {
                double a = (double)tab[dy[t * n + i]];     /* dY^T[i, t] = dY[t, i] */
                const uint16_t *xrow = x + t * k;
                for (int64_t j = 0; j < k; ++j) acc[j] += a * (double)tab[xrow[j]];
            }
            for (int64_t j = 0; j < k; ++j) dw[ii * k + j] = oracle_encode16_rne(acc[j], is_bf16);
        }
        free(acc);
    }
    if (err == OR_OK && db) {
#pragma omp parallel for
        for (int64_t i = 0; i < n; ++i) {
            double s = 0.0;
            for (int64_t t = 0; t < m; ++t) s += (double)tab[dy[t * n + i]];
            db[i] = oracle_encode16_rne(s, is_bf16);
        }
    }
    free(tab);
    return err;
}

/* ------------------------------------------------------------------------ */
/* [QAR] Low-bit element formats, decoded from their definitions.             */
/*   FP8 E4M3FN: 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent 0 is  */
/*   subnormal (m/8 * 2^-6); no infinities; S.1111.111 is NaN.                */
/*   FP8 E5M2: 1 sign, 5 exponent (bias 15), 2 mantissa bits; exponent 0 is   */
/*   subnormal (m/4 * 2^-14); exponent 31 is inf (m = 0) or NaN.              */
/*   E8M0 (mx scale): an unsigned biased exponent, 2^(e - 127); 0xFF is NaN.  */
/* ------------------------------------------------------------------------ */
double oracle_decode_fp8(uint8_t v, int is_e5m2) {
    int sign = (v >> 7) & 1;
    int e, m;
    double mag;
    if (is_e5m2) {
        e = (v >> 2) & 0x1F;
        m = v & 0x3;
        if (e == 31) return m == 0 ? (sign ? -INFINITY : INFINITY) : NAN;
        mag = e == 0 ? ldexp((double)m / 4.0, -14) : ldexp(1.0 + (double)m / 4.0, e - 15);
    } else {
        e = (v >> 3) & 0xF;
        m = v & 0x7;
        if (e == 15 && m == 7) return NAN;
        mag = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    }
    return sign ? -mag : mag;
}

double oracle_decode_e8m0(uint8_t v) {
    if (v == 0xFF) return NAN;
    return ldexp(1.0, (int)v - 127);
}

/* ------------------------------------------------------------------------ */
/* [QAR] QuantAllReduce:  AllGatherData = AllGather(x),                       */
/*   AllGatherScales = AllGather(scales),                                     */
/*   output = Reduce(AllGatherScales * AllGatherData), Reduce = sum over the  */
/*   ranks (reduceOp "sum").  Rank r's x_r (bs, h) and scales_r are given     */
/* side by side; every rank receives the same output (bs, h):                 */
/*   out[t, j] = sum_r dec(x_r[t, j]) * dec(scales_r[t, j / G])               */
/*   x_kind 0 int8, 1 fp8 e4m3fn, 2 fp8 e5m2                                  */
/*   scale_kind 0: fp32, one per token per group of G = 128 (pertoken-        */
/*     pergroup, scales (bs, h/128));  1: e8m0, one per group of G = 32 (mx,  */
/*     scales (bs, h/64, 2) read flat as (bs, h/32)).                         */
/*   out_kind 0 fp32, 1 fp16, 2 bf16.                                         */
/* Reading: the products are exact in fp64 (at most 8 + 24 significant      */
/* bits), summed in fp64 in rank order and rounded once, nearest-even, to    */
/* the output type.                                                           */
/* ------------------------------------------------------------------------ */
int oracle_quant_all_reduce(const uint8_t *const *x_chunks, const void *const *scale_chunks, int world_size,
                            int64_t bs, int64_t h, int x_kind, int scale_kind, int out_kind, void *out) {
    if (!x_chunks || !scale_chunks || !out || world_size < 1 || bs < 1 || h < 1) return OR_ERR_ARG;
    if (x_kind < 0 || x_kind > 2 || scale_kind < 0 || scale_kind > 1 || out_kind < 0 || out_kind > 2)
        return OR_ERR_ARG;
    int64_t G = scale_kind == 0 ? 128 : 32;
    if (h % G != 0) return OR_ERR_ARG;
    int64_t groups = h / G;
#pragma omp parallel for
    for (int64_t t = 0; t < bs; ++t) {
        for (int64_t j = 0; j < h; ++j) {
            double s = 0.0;
            for (int r = 0; r < world_size; ++r) {
                uint8_t xv = x_chunks[r][t * h + j];
                double x = x_kind == 0 ? (double)(int8_t)xv : oracle_decode_fp8(xv, x_kind == 2);
                double sc = scale_kind == 0 ? (double)((const float *)scale_chunks[r])[t * groups + j / G]
                                            : oracle_decode_e8m0(((const uint8_t *)scale_chunks[r])[t * groups + j / G]);
                s += x * sc;
            }
            if (out_kind == 0)
                ((float *)out)[t * h + j] = (float)s;
            else
                ((uint16_t *)out)[t * h + j] = oracle_encode16_rne(s, out_kind == 2);
        }
    }
    return OR_OK;
}
