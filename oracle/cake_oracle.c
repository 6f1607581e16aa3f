/*
 * cake_oracle.c -- plain, single-threaded FP64 reference of the training
 * RMSNorm forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline / reference arm do.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * What it computes (the pages print no formula, so the definitions below are
 * the standard RMSNorm and its exact gradient; the dtypes and the output list
 * follow the pages):
 *   - outputs and dtypes: y (BF16) and rstd (FP32) from the forward, dx (BF16)
 *     and dw (FP32) from the backward -- "Speedups ... GB300 windows" commit
 *     (#8577) quoted on the page of PR #8208, intro; restated on PR #8899's
 *     page, first paragraph.
 *   - fused residual add: the residual route also returns the BF16 sum h_new
 *     and normalises it -- #8577 commit, "Key" (`res`).
 *   - per-head views [T,24,256] with strides (12288,512,1) and [T,4,256] with
 *     one shared w[256]: PR #8208 page, description.
 *   - dw is checked against an FP64 result computed at the kernel's FP32
 *     rstd: PR #8208 page, description.  So every function here that produces y, dx or dw takes the
 *     rstd to use as an input (the kernel's FP32 value, widened to double).
 *
 * Row r of a [T, nh, H] view is (t, k) = (r / nh, r % nh); element j of that
 * row sits at base + t*stride_t + k*stride_h + j.  Plain [T, H] rows are the
 * nh = 1 case.
 *
 * Per row, in FP64, j ascending:
 *   h_j     = x_j                       (no residual)
 *   h_j     = RNE_bf16(x_j + res_j)     (residual; the sum of two BF16 values
 *                                        is exact in FP64)
 *   ms      = (1/H) sum_j h_j^2
 *   rstd64  = 1 / sqrt(ms + eps)
 *   y_j     = h_j * rs * w_j            (rs = the rstd handed in, else rstd64)
 * Backward, per row, with rs the kernel's rstd:
 *   g_j  = dy_j * w_j,   xh_j = h_j * rs,   c = (1/H) sum_j g_j * xh_j
 *   dx_j = rs * (g_j - xh_j * c)  [+ dh_j, the gradient that reaches h_new
 *                                   directly on the residual route]
 * and over all rows, r ascending (the exact-order FP64 column sum):
 *   dw_j = sum_r dy_rj * h_rj * rs_r
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ---- BF16 <-> FP64 ----------------------------------------------------- */

static double bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round an FP64 value to the nearest BF16 value, ties to even, in one step
 * (no intermediate FP32 rounding).  BF16 keeps 8 significant bits, has the
 * FP32 exponent range, subnormal spacing 2^-133 and largest finite value
 * (2 - 2^-7) * 2^127. */
static uint16_t f64_to_bf16_rne(double v)
{
    if (isnan(v))
        return 0x7fc0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7f80;
    int e;
    frexp(a, &e);            /* a in [2^(e-1), 2^e) */
    int q = e - 8;           /* spacing of 8-bit significands in that binade */
    if (q < -133)
        q = -133;            /* subnormal range */
    double r = nearbyint(ldexp(a, -q)); /* default mode: ties to even */
    double out = ldexp(r, q);
    const double max_bf16 = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
    if (out > max_bf16)
        return sign | 0x7f80;
    float f = (float)out;    /* exact: at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

static double weight_at(const void *w, int w_is_f32, int64_t j)
{
    if (w_is_f32)
        return (double)((const float *)w)[j];
    return bf16_to_f64(((const uint16_t *)w)[j]);
}

static int64_t row_offset(int64_t r, int64_t nh, int64_t st, int64_t sh)
{
    int64_t t = r / nh, k = r % nh;
    return t * st + k * sh;
}

/* ---- per-row kernels of the definition, on FP64 rows ------------------- */

static double row_rstd64(const double *h, int64_t H, double eps)
{
    double ss = 0.0;
    for (int64_t j = 0; j < H; ++j)
        ss += h[j] * h[j];
    double ms = ss / (double)H;
    return 1.0 / sqrt(ms + eps);
}

static void row_y(const double *h, const double *w, int64_t H, double rs, double *y)
{
    for (int64_t j = 0; j < H; ++j)
        y[j] = h[j] * rs * w[j];
}

static void row_dx(const double *dy, const double *h, const double *w,
                   const double *dh, int64_t H, double rs, double *dx)
{
    double c = 0.0;
    for (int64_t j = 0; j < H; ++j)
        c += (dy[j] * w[j]) * (h[j] * rs);
    c /= (double)H;
    for (int64_t j = 0; j < H; ++j) {
        double g = dy[j] * w[j];
        double xh = h[j] * rs;
        dx[j] = rs * (g - xh * c) + (dh ? dh[j] : 0.0);
    }
}

/* ---- FP64-array entry points (finite-difference and invariant checks) -- */

/* rows [R][H] contiguous.  rstd_in may be NULL (then rstd64 is used for y). */
ORACLE_API int cake_oracle_fwd_f64(int64_t R, int64_t H, const double *h,
                                   const double *w, double eps,
                                   const double *rstd_in, double *y,
                                   double *rstd64)
{
    if (R < 0 || H <= 0 || !h || !w || !y || !rstd64)
        return 1;
    for (int64_t r = 0; r < R; ++r) {
        const double *hr = h + r * H;
        rstd64[r] = row_rstd64(hr, H, eps);
        double rs = rstd_in ? rstd_in[r] : rstd64[r];
        row_y(hr, w, H, rs, y + r * H);
    }
    return 0;
}

/* dx [R][H] and dw [H]; dh may be NULL. */
ORACLE_API int cake_oracle_bwd_f64(int64_t R, int64_t H, const double *dy,
                                   const double *h, const double *rstd,
                                   const double *w, const double *dh,
                                   double *dx, double *dw)
{
    if (R < 0 || H <= 0 || !dy || !h || !rstd || !w || !dx || !dw)
        return 1;
    for (int64_t r = 0; r < R; ++r)
        row_dx(dy + r * H, h + r * H, w, dh ? dh + r * H : NULL, H, rstd[r],
               dx + r * H);
    for (int64_t j = 0; j < H; ++j) {
        double s = 0.0;
        for (int64_t r = 0; r < R; ++r)
            s += dy[r * H + j] * h[r * H + j] * rstd[r];
        dw[j] = s;
    }
    return 0;
}

/* ---- BF16-storage entry points over strided [T, nh, H] views ----------- */

/* Decode row r of a BF16 view into FP64. */
static void load_row(const uint16_t *base, int64_t r, int64_t nh, int64_t st,
                     int64_t sh, int64_t H, double *out)
{
    const uint16_t *p = base + row_offset(r, nh, st, sh);
    for (int64_t j = 0; j < H; ++j)
        out[j] = bf16_to_f64(p[j]);
}

/* h = x (no residual) or h = RNE_bf16(x + res); h_bits receives the BF16 bits. */
static void load_h(const uint16_t *x, int64_t x_st, int64_t x_sh,
                   const uint16_t *res, int64_t res_st, int64_t res_sh,
                   int64_t r, int64_t nh, int64_t H, double *h, double *tmp,
                   uint16_t *h_bits)
{
    load_row(x, r, nh, x_st, x_sh, H, h);
    if (res) {
        load_row(res, r, nh, res_st, res_sh, H, tmp);
        for (int64_t j = 0; j < H; ++j) {
            uint16_t b = f64_to_bf16_rne(h[j] + tmp[j]);
            if (h_bits)
                h_bits[j] = b;
            h[j] = bf16_to_f64(b);
        }
    } else if (h_bits) {
        const uint16_t *p = x + row_offset(r, nh, x_st, x_sh);
        for (int64_t j = 0; j < H; ++j)
            h_bits[j] = p[j];
    }
}

/*
 * Forward over the listed rows (rows == NULL: all T*nh rows, in order).
 * Outputs are packed [nrows][H] / [nrows]:
 *   y      FP64 values of h * rs * w (rs = rstd_in[row] if rstd_in, else rstd64)
 *   rstd64 FP64 1/sqrt(mean(h^2) + eps)
 *   h_new  BF16 bits of h (may be NULL)
 * work must hold 3*H doubles.
 */
ORACLE_API int cake_oracle_fwd_rows(int64_t T, int64_t nh, int64_t H,
                                    const uint16_t *x, int64_t x_st, int64_t x_sh,
                                    const uint16_t *res, int64_t res_st, int64_t res_sh,
                                    const void *w, int w_is_f32, double eps,
                                    const float *rstd_in, const int64_t *rows,
                                    int64_t nrows, double *y, double *rstd64,
                                    uint16_t *h_new, double *work)
{
    if (T < 0 || nh <= 0 || H <= 0 || !x || !w || !work)
        return 1;
    if (!rows)
        nrows = T * nh;
    double *h = work, *tmp = work + H, *wd = work + 2 * H;
    for (int64_t j = 0; j < H; ++j)
        wd[j] = weight_at(w, w_is_f32, j);
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        if (r < 0 || r >= T * nh)
            return 2;
        load_h(x, x_st, x_sh, res, res_st, res_sh, r, nh, H, h, tmp,
               h_new ? h_new + i * H : NULL);
        double r64 = row_rstd64(h, H, eps);
        if (rstd64)
            rstd64[i] = r64;
        if (y)
            row_y(h, wd, H, rstd_in ? (double)rstd_in[r] : r64, y + i * H);
    }
    return 0;
}

/*
 * Backward dx over the listed rows (rows == NULL: all rows).  h is the
 * normalised input (x, or the saved h_new on the residual route); rstd is the
 * kernel's FP32 rstd per row; dh (nullable) is the gradient reaching h_new.
 * dx is packed [nrows][H] FP64.  work must hold 4*H doubles.
 */
ORACLE_API int cake_oracle_bwd_rows(int64_t T, int64_t nh, int64_t H,
                                    const uint16_t *dy, int64_t dy_st, int64_t dy_sh,
                                    const uint16_t *h, int64_t h_st, int64_t h_sh,
                                    const float *rstd, const void *w, int w_is_f32,
                                    const uint16_t *dh, int64_t dh_st, int64_t dh_sh,
                                    const int64_t *rows, int64_t nrows, double *dx,
                                    double *work)
{
    if (T < 0 || nh <= 0 || H <= 0 || !dy || !h || !rstd || !w || !dx || !work)
        return 1;
    if (!rows)
        nrows = T * nh;
    double *dyr = work, *hr = work + H, *dhr = work + 2 * H, *wd = work + 3 * H;
    for (int64_t j = 0; j < H; ++j)
        wd[j] = weight_at(w, w_is_f32, j);
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        if (r < 0 || r >= T * nh)
            return 2;
        load_row(dy, r, nh, dy_st, dy_sh, H, dyr);
        load_row(h, r, nh, h_st, h_sh, H, hr);
        if (dh)
            load_row(dh, r, nh, dh_st, dh_sh, H, dhr);
        row_dx(dyr, hr, wd, dh ? dhr : NULL, H, (double)rstd[r], dx + i * H);
    }
    return 0;
}

/*
 * dw for the listed columns (cols == NULL: all H columns): the FP64 sum over
 * every row, r ascending, of dy_rj * h_rj * rstd_r.
 */
ORACLE_API int cake_oracle_dw_cols(int64_t T, int64_t nh, int64_t H,
                                   const uint16_t *dy, int64_t dy_st, int64_t dy_sh,
                                   const uint16_t *h, int64_t h_st, int64_t h_sh,
                                   const float *rstd, const int64_t *cols,
                                   int64_t ncols, double *dw)
{
    if (T < 0 || nh <= 0 || H <= 0 || !dy || !h || !rstd || !dw)
        return 1;
    if (!cols)
        ncols = H;
    for (int64_t i = 0; i < ncols; ++i) {
        int64_t j = cols ? cols[i] : i;
        if (j < 0 || j >= H)
            return 2;
        dw[i] = 0.0;
    }
    const int64_t R = T * nh;
    for (int64_t r = 0; r < R; ++r) {
        const uint16_t *dyr = dy + row_offset(r, nh, dy_st, dy_sh);
        const uint16_t *hr = h + row_offset(r, nh, h_st, h_sh);
        double rs = (double)rstd[r];
        for (int64_t i = 0; i < ncols; ++i) {
            int64_t j = cols ? cols[i] : i;
            dw[i] += bf16_to_f64(dyr[j]) * bf16_to_f64(hr[j]) * rs;
        }
    }
    return 0;
}

/* RNE rounding of FP64 values to BF16 bits (used to state "within 1 BF16 ulp
 * of the FP64 value rounded"). */
ORACLE_API void cake_oracle_bf16_round(const double *v, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = f64_to_bf16_rne(v[i]);
}
