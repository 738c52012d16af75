/*
 * FP64 reference ("oracle") for RMSNorm forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this file;
 * only the tests, the package's smoke check and the bench's CPU baseline do.
 * It shares no code, header or constant with the CUDA library.
 *
 * What it computes is the plain definition, on rows given in canonical
 * logical order (inactive/padding rows are simply absent):
 *
 *   ms_g    = (1/H) * sum_h x_gh^2
 *   rstd_g  = 1 / sqrt(ms_g + eps)                       (eps inside the root)
 *   xhat_gh = x_gh * rstd_g
 *   y_gh    = xhat_gh * w_h                               (forward)
 *   g_gh    = dy_gh * w_h
 *   m_g     = (1/H) * sum_h g_gh * xhat_gh
 *   dx_gh   = rstd_g * (g_gh - xhat_gh * m_g)             (VJP of y w.r.t. x)
 *   dw_h    = sum_g dy_gh * xhat_gh                       (VJP of y w.r.t. w)
 *
 * Sources: "[WS1 Closeout][Backward] Reusable gradient-invariance harness
 * and operator adapters" (RL-Kernel issue #270), Goal/Scope and "Required
 * adapters: RMSNorm dx/dweight"; "WS1 C4 (#270) closeout evidence",
 * "Historical finding - RMSNorm dweight is not chunk/batch decomposable"
 * (the weight gradient is a sum of per-logical-row FP32 contributions
 * dy * xhat over the active rows; inactive tokens contribute 0).  The closed
 * forms y = x*w/sqrt(mean(x^2)+eps) and dweight = sum_rows dy*xhat are the
 * benchmark statement's; dx is the derivative of that closed form.
 *
 * Besides the values it returns two error scales used by the tests'
 * tolerances: per element dx_scale = rstd*(|g| + |xhat*m|) (the size of the
 * two terms that cancel in dx) and per column dw_scale = sqrt(sum_g c_g^2)
 * with c = dy*xhat (the root-sum-square of the terms of dweight).
 *
 * Plain loops, no blocking, no vectorisation pragmas, built without
 * fast-math.  Inputs are bf16 bit patterns converted exactly to double, or
 * doubles directly (for finite-difference checks).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* bf16 is the top half of an IEEE binary32: widen by 16 zero bits. */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

void oracle_bf16_array_to_double(const uint16_t *src, int64_t n, double *dst)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = oracle_bf16_to_double(src[i]);
}

/* Forward on one row: returns rstd, writes y (may be NULL). */
static double row_forward(const double *x, const double *w, int64_t H, double eps, double *y)
{
    double ss = 0.0;
    for (int64_t h = 0; h < H; ++h)
        ss += x[h] * x[h];
    double ms = ss / (double)H;
    double rstd = 1.0 / sqrt(ms + eps);
    if (y)
        for (int64_t h = 0; h < H; ++h)
            y[h] = (x[h] * rstd) * w[h];
    return rstd;
}

/* y [n,H] and rstd [n] (either may be NULL) from x [n,H], w [H]. */
void oracle_rmsnorm_fwd_f64(const double *x, const double *w, int64_t n, int64_t H,
                            double eps, double *y, double *rstd)
{
    for (int64_t g = 0; g < n; ++g) {
        double r = row_forward(x + g * H, w, H, eps, y ? y + g * H : NULL);
        if (rstd)
            rstd[g] = r;
    }
}

/*
 * Backward over n logical rows.  dx, dx_scale: [n,H] (may be NULL);
 * dweight, dw_scale: [H] (may be NULL).  dweight sums over all n rows.
 */
void oracle_rmsnorm_bwd_f64(const double *x, const double *w, const double *dy,
                            int64_t n, int64_t H, double eps,
                            double *dx, double *dx_scale, double *dweight, double *dw_scale)
{
    if (dweight)
        for (int64_t h = 0; h < H; ++h) dweight[h] = 0.0;
    if (dw_scale)
        for (int64_t h = 0; h < H; ++h) dw_scale[h] = 0.0;

    for (int64_t g = 0; g < n; ++g) {
        const double *xr = x + g * H;
        const double *dyr = dy + g * H;
        double rstd = row_forward(xr, w, H, eps, NULL);

        double dot = 0.0;                       /* sum_h g_h * xhat_h */
        for (int64_t h = 0; h < H; ++h)
            dot += (dyr[h] * w[h]) * (xr[h] * rstd);
        double m = dot / (double)H;

        for (int64_t h = 0; h < H; ++h) {
            double xhat = xr[h] * rstd;
            double gh = dyr[h] * w[h];
            if (dx)
                dx[g * H + h] = rstd * (gh - xhat * m);
            if (dx_scale)
                dx_scale[g * H + h] = rstd * (fabs(gh) + fabs(xhat * m));
            double c = dyr[h] * xhat;
            if (dweight)
                dweight[h] += c;
            if (dw_scale)
                dw_scale[h] += c * c;
        }
    }
    if (dw_scale)
        for (int64_t h = 0; h < H; ++h) dw_scale[h] = sqrt(dw_scale[h]);
}

/* bf16 entry points: rows are converted exactly to double one at a time. */
void oracle_rmsnorm_fwd_bf16(const uint16_t *x, const uint16_t *w, int64_t n, int64_t H,
                             double eps, double *y, double *rstd, double *scratch /* [2H] */)
{
    double *wd = scratch, *xd = scratch + H;
    oracle_bf16_array_to_double(w, H, wd);
    for (int64_t g = 0; g < n; ++g) {
        oracle_bf16_array_to_double(x + g * H, H, xd);
        oracle_rmsnorm_fwd_f64(xd, wd, 1, H, eps, y ? y + g * H : NULL, rstd ? rstd + g : NULL);
    }
}

void oracle_rmsnorm_bwd_bf16(const uint16_t *x, const uint16_t *w, const uint16_t *dy,
                             int64_t n, int64_t H, double eps,
                             double *dx, double *dx_scale, double *dweight, double *dw_scale,
                             double *scratch /* [5H] */)
{
    double *wd = scratch, *xd = scratch + H, *dyd = scratch + 2 * H;
    double *dwrow = scratch + 3 * H, *dsrow = scratch + 4 * H;
    oracle_bf16_array_to_double(w, H, wd);
    if (dweight)
        for (int64_t h = 0; h < H; ++h) dweight[h] = 0.0;
    if (dw_scale)
        for (int64_t h = 0; h < H; ++h) dw_scale[h] = 0.0;
    for (int64_t g = 0; g < n; ++g) {
        oracle_bf16_array_to_double(x + g * H, H, xd);
        oracle_bf16_array_to_double(dy + g * H, H, dyd);
        oracle_rmsnorm_bwd_f64(xd, wd, dyd, 1, H, eps,
                               dx ? dx + g * H : NULL, dx_scale ? dx_scale + g * H : NULL,
                               dwrow, dsrow);
        for (int64_t h = 0; h < H; ++h) {
            if (dweight) dweight[h] += dwrow[h];
            if (dw_scale) dw_scale[h] += dsrow[h] * dsrow[h];
        }
    }
    if (dw_scale)
        for (int64_t h = 0; h < H; ++h) dw_scale[h] = sqrt(dw_scale[h]);
}
