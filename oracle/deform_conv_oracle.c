/*
 * Deformable convolution oracle: plain, slow, fp64 CPU statement of the layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file; only the test suite, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or constant with the CUDA
 * library.
 *
 * Source of every step: the explainer page "DefT: Boosting Scalability of
 * Deformable Convolution Operations on GPUs" (ASPLOS 2023).
 *   - "The argument in one glance / What people did": the layer is three
 *     operators run back to back -- an offset convolution, a bilinear
 *     interpolation that builds the deformed feature map, and the main
 *     convolution over that map.
 *   - "Following a deformable layer through DefT", Step 1 of 5: the offset
 *     convolution produces, for every filter position at every output location,
 *     a fractional (y, x) offset; it is added to the base sampling coordinate and
 *     the sample falls among four neighbouring pixels.
 *   - "The argument in one glance / Why it fell short": the four neighbours are
 *     blended by their bilinear weights.
 *   Written out, y(p0) = sum_k w_k * x(p0 + p_k + dp_k) with x read by bilinear
 *   interpolation and every corner outside the image contributing zero.
 *
 * Readings where the page is silent (each one is listed with its reason in the
 * design notes of the repository):
 *   - the offset convolution has the main convolution's kernel size, stride,
 *     padding and dilation, plus a bias, so its output grid is the output grid;
 *   - offset channel 2*(g*K + k) is the row shift dy and 2*(g*K + k) + 1 the
 *     column shift dx of tap k = i*Kw + j in offset group g;
 *   - input channel c belongs to offset group c / (C_in / G);
 *   - corners outside [0,H) x [0,W) contribute zero, with no clamping;
 *   - at an integer coordinate the lower corner is floor(p), so the derivative
 *     of the sample with respect to p is the right-sided difference;
 *   - floor(p) is an integer decision, so it is taken on the float32 value of
 *     the coordinate, the precision the GPU kernels form it in (orc_cell).
 *
 * The backward pass is the exact derivative of that definition, written out
 * step by step in fp64.  Loops are parallelised with OpenMP only over indices
 * whose outputs are disjoint; no blocking, fusion or reordering of the sums
 * beyond that.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int n, c_in, h, w, c_out, kh, kw;
  int stride_h, stride_w, pad_h, pad_w, dil_h, dil_w;
  int groups;
} orc_problem;

#define ORC_OK 0
#define ORC_BAD_ARG 1
#define ORC_NO_MEMORY 2

static int orc_out_h(const orc_problem *p) {
  return (p->h + 2 * p->pad_h - p->dil_h * (p->kh - 1) - 1) / p->stride_h + 1;
}
static int orc_out_w(const orc_problem *p) {
  return (p->w + 2 * p->pad_w - p->dil_w * (p->kw - 1) - 1) / p->stride_w + 1;
}

int orc_check(const orc_problem *p) {
  if (!p) return ORC_BAD_ARG;
  if (p->n <= 0 || p->c_in <= 0 || p->h <= 0 || p->w <= 0 || p->c_out <= 0 ||
      p->kh <= 0 || p->kw <= 0 || p->stride_h <= 0 || p->stride_w <= 0 ||
      p->pad_h < 0 || p->pad_w < 0 || p->dil_h <= 0 || p->dil_w <= 0 ||
      p->groups <= 0 || p->c_in % p->groups != 0)
    return ORC_BAD_ARG;
  if (p->h + 2 * p->pad_h - p->dil_h * (p->kh - 1) - 1 < 0) return ORC_BAD_ARG;
  if (p->w + 2 * p->pad_w - p->dil_w * (p->kw - 1) - 1 < 0) return ORC_BAD_ARG;
  return ORC_OK;
}

/* Pixel (a, b) of one H x W plane, zero outside the image. */
static double orc_pixel(const double *plane, int H, int W, long a, long b) {
  if (a < 0 || a >= H || b < 0 || b >= W) return 0.0;
  return plane[a * (long)W + b];
}

/* Whether (py, px) can touch the image at all.  Outside this box every one of
 * the four corners is outside the image, so the sample and both of its
 * derivatives are zero; the guard also keeps floor() finite.  NaN is outside. */
static int orc_near_image(int H, int W, double py, double px) {
  return py > -2.0 && py < (double)H + 1.0 && px > -2.0 && px < (double)W + 1.0;
}

/* Bilinear sample of one plane at the fractional point (py, px), written as
 * the blend of the four neighbouring pixels ("Why it fell short").  The cell
 * (lower corner) is (cy, cx); the plain definition takes cy = floor(py),
 * cx = floor(px), which is what orc_bilinear below does. */
static double orc_bilinear_cell(const double *plane, int H, int W, double py,
                                double px, double cy, double cx) {
  long a = (long)cy, b = (long)cx;
  double ly = py - cy, lx = px - cx;
  double hy = 1.0 - ly, hx = 1.0 - lx;
  return hy * hx * orc_pixel(plane, H, W, a, b) +
         hy * lx * orc_pixel(plane, H, W, a, b + 1) +
         ly * hx * orc_pixel(plane, H, W, a + 1, b) +
         ly * lx * orc_pixel(plane, H, W, a + 1, b + 1);
}

double orc_bilinear(const double *plane, int H, int W, double py, double px) {
  if (!orc_near_image(H, W, py, px)) return 0.0;
  return orc_bilinear_cell(plane, H, W, py, px, floor(py), floor(px));
}

/* The same sample as a sum over every pixel of the image with the triangular
 * (tent) kernel max(0, 1-|py-a|) * max(0, 1-|px-b|).  Pixels outside the image
 * are simply absent from the sum.  Independent of orc_bilinear on purpose. */
double orc_bilinear_closed_form(const double *plane, int H, int W, double py,
                                double px) {
  double s = 0.0;
  for (int a = 0; a < H; ++a) {
    double ky = 1.0 - fabs(py - (double)a);
    if (!(ky > 0.0)) continue;
    for (int b = 0; b < W; ++b) {
      double kx = 1.0 - fabs(px - (double)b);
      if (!(kx > 0.0)) continue;
      s += ky * kx * plane[(long)a * W + b];
    }
  }
  return s;
}

/* Derivatives of the bilinear sample with respect to py and px inside the
 * cell (cy, cx) (with cy = floor(py): right-sided difference at integers). */
static void orc_bilinear_grad_cell(const double *plane, int H, int W, double py,
                                   double px, double cy, double cx,
                                   double *d_py, double *d_px) {
  long a = (long)cy, b = (long)cx;
  double ly = py - cy, lx = px - cx;
  double v00 = orc_pixel(plane, H, W, a, b);
  double v01 = orc_pixel(plane, H, W, a, b + 1);
  double v10 = orc_pixel(plane, H, W, a + 1, b);
  double v11 = orc_pixel(plane, H, W, a + 1, b + 1);
  *d_py = (1.0 - lx) * (v10 - v00) + lx * (v11 - v01);
  *d_px = (1.0 - ly) * (v01 - v00) + ly * (v11 - v10);
}

void orc_bilinear_grad(const double *plane, int H, int W, double py, double px,
                       double *d_py, double *d_px) {
  *d_py = 0.0;
  *d_px = 0.0;
  if (!orc_near_image(H, W, py, px)) return;
  orc_bilinear_grad_cell(plane, H, W, py, px, floor(py), floor(px), d_py, d_px);
}

/* Adjoint of the sample with respect to the plane: adds g times each corner's
 * weight to that corner, for the corners inside the image. */
static void orc_bilinear_scatter_cell(double *plane, int H, int W, double py,
                                      double px, double cy, double cx, double g) {
  long a = (long)cy, b = (long)cx;
  double ly = py - cy, lx = px - cx;
  double hy = 1.0 - ly, hx = 1.0 - lx;
  long ya[2] = {a, a + 1}, xb[2] = {b, b + 1};
  double wy[2] = {hy, ly}, wx[2] = {hx, lx};
  for (int u = 0; u < 2; ++u)
    for (int v = 0; v < 2; ++v) {
      if (ya[u] < 0 || ya[u] >= H || xb[v] < 0 || xb[v] >= W) continue;
      plane[ya[u] * W + xb[v]] += wy[u] * wx[v] * g;
    }
}

/* Cell of a sampling coordinate base + shift.  floor() turns the coordinate
 * into an integer (which four pixels are blended, and on which side of a
 * pixel line the derivative is taken), so that decision is made in the
 * precision the GPU kernels form the coordinate in: float32, on
 * fl32(fl32(base) + fl32(shift)).  The weights inside the cell stay fp64.
 * Away from pixel lines this is floor(base + shift) exactly; within a float32
 * rounding of a line it picks the same side as the kernels. */
double orc_cell(long base, double shift) {
  float p32 = (float)base + (float)shift;
  return floor((double)p32);
}

/* Step 1 of 5: offset convolution.
 * off[n, m, ho, wo] = b_off[m] + sum_{c,i,j} w_off[m, c, i, j] *
 *                     xbar[n, c, ho*s - pad + i*dil, wo*s - pad + j*dil]
 *                     (+ offset_add[n, m, ho, wo])
 * with xbar zero outside the image and m in [0, 2*G*Kh*Kw).  b_off and
 * offset_add may be NULL (taken as zero). */
int orc_offsets(const orc_problem *p, const double *x, const double *w_off,
                const double *b_off, const double *offset_add, double *off) {
  int rc = orc_check(p);
  if (rc) return rc;
  const int Ho = orc_out_h(p), Wo = orc_out_w(p);
  const int K = p->kh * p->kw, M = 2 * p->groups * K;
  const long HW = (long)p->h * p->w, HoWo = (long)Ho * Wo;
#pragma omp parallel for collapse(2) schedule(static)
  for (int n = 0; n < p->n; ++n)
    for (int m = 0; m < M; ++m)
      for (int ho = 0; ho < Ho; ++ho)
        for (int wo = 0; wo < Wo; ++wo) {
          double s = b_off ? b_off[m] : 0.0;
          for (int c = 0; c < p->c_in; ++c) {
            const double *plane = x + ((long)n * p->c_in + c) * HW;
            for (int i = 0; i < p->kh; ++i)
              for (int j = 0; j < p->kw; ++j) {
                long a = (long)ho * p->stride_h - p->pad_h + (long)i * p->dil_h;
                long b = (long)wo * p->stride_w - p->pad_w + (long)j * p->dil_w;
                s += w_off[(((long)m * p->c_in + c) * p->kh + i) * p->kw + j] *
                     orc_pixel(plane, p->h, p->w, a, b);
              }
          }
          long o = ((long)n * M + m) * HoWo + (long)ho * Wo + wo;
          if (offset_add) s += offset_add[o];
          off[o] = s;
        }
  return ORC_OK;
}

/* Sampling point of tap (i, j) at output (ho, wo) of image n for offset
 * group g: base grid position plus the learned shift (Step 1 of 5).  Returns
 * 0 when no corner can touch the image (sample and derivatives are zero),
 * else 1 with the point (py, px) and its cell (cy, cx). */
static int orc_sample_point(const orc_problem *p, const double *off, int n,
                            int g, int i, int j, int ho, int wo, double *py,
                            double *px, double *cy, double *cx) {
  const int Ho = orc_out_h(p), Wo = orc_out_w(p);
  const int K = p->kh * p->kw, M = 2 * p->groups * K;
  const int k = i * p->kw + j;
  const long HoWo = (long)Ho * Wo;
  const long base = (long)n * M * HoWo + (long)ho * Wo + wo;
  double dy = off[base + (long)(2 * (g * K + k)) * HoWo];
  double dx = off[base + (long)(2 * (g * K + k) + 1) * HoWo];
  long by = (long)ho * p->stride_h - p->pad_h + (long)i * p->dil_h;
  long bx = (long)wo * p->stride_w - p->pad_w + (long)j * p->dil_w;
  *py = (double)by + dy;
  *px = (double)bx + dx;
  if (!orc_near_image(p->h, p->w, *py, *px)) return 0;
  *cy = orc_cell(by, dy);
  *cx = orc_cell(bx, dx);
  return 1;
}

/* The deformed ("unrolled") feature map, col[n, c, k, ho, wo] = bilinear
 * sample of channel c at tap k's displaced point ("What people did before,
 * and where it broke": the interpolation's output). */
int orc_column(const orc_problem *p, const double *x, const double *off,
               double *col) {
  int rc = orc_check(p);
  if (rc) return rc;
  const int Ho = orc_out_h(p), Wo = orc_out_w(p);
  const int K = p->kh * p->kw, Cg = p->c_in / p->groups;
  const long HW = (long)p->h * p->w, HoWo = (long)Ho * Wo;
#pragma omp parallel for collapse(2) schedule(static)
  for (int n = 0; n < p->n; ++n)
    for (int c = 0; c < p->c_in; ++c) {
      const double *plane = x + ((long)n * p->c_in + c) * HW;
      const int g = c / Cg;
      for (int i = 0; i < p->kh; ++i)
        for (int j = 0; j < p->kw; ++j) {
          const int k = i * p->kw + j;
          double *dst = col + (((long)n * p->c_in + c) * K + k) * HoWo;
          for (int ho = 0; ho < Ho; ++ho)
            for (int wo = 0; wo < Wo; ++wo) {
              double py, px, cy, cx;
              double v = 0.0;
              if (orc_sample_point(p, off, n, g, i, j, ho, wo, &py, &px, &cy, &cx))
                v = orc_bilinear_cell(plane, p->h, p->w, py, px, cy, cx);
              dst[(long)ho * Wo + wo] = v;
            }
        }
    }
  return ORC_OK;
}

/* Adjoint of orc_column with respect to x: gx[n, c] += sum over taps and
 * outputs of gcol times the corner weights.  gx is overwritten. */
int orc_column_adjoint(const orc_problem *p, const double *off,
                       const double *gcol, double *gx) {
  int rc = orc_check(p);
  if (rc) return rc;
  const int Ho = orc_out_h(p), Wo = orc_out_w(p);
  const int K = p->kh * p->kw, Cg = p->c_in / p->groups;
  const long HW = (long)p->h * p->w, HoWo = (long)Ho * Wo;
#pragma omp parallel for collapse(2) schedule(static)
  for (int n = 0; n < p->n; ++n)
    for (int c = 0; c < p->c_in; ++c) {
      double *plane = gx + ((long)n * p->c_in + c) * HW;
      memset(plane, 0, sizeof(double) * HW);
      const int g = c / Cg;
      for (int i = 0; i < p->kh; ++i)
        for (int j = 0; j < p->kw; ++j) {
          const int k = i * p->kw + j;
          const double *src = gcol + (((long)n * p->c_in + c) * K + k) * HoWo;
          for (int ho = 0; ho < Ho; ++ho)
            for (int wo = 0; wo < Wo; ++wo) {
              double py, px, cy, cx;
              if (orc_sample_point(p, off, n, g, i, j, ho, wo, &py, &px, &cy, &cx))
                orc_bilinear_scatter_cell(plane, p->h, p->w, py, px, cy, cx,
                                          src[(long)ho * Wo + wo]);
            }
        }
    }
  return ORC_OK;
}

/* Forward pass of the whole layer.
 * off = offset convolution (+ offset_add); col = deformed map;
 * y[n, o, ho, wo] = sum_{c, k} w[o, c, k] * col[n, c, k, ho, wo].
 * offset_out may be NULL. */
int orc_forward(const orc_problem *p, const double *x, const double *w_off,
                const double *b_off, const double *w, const double *offset_add,
                double *y, double *offset_out) {
  int rc = orc_check(p);
  if (rc) return rc;
  const int Ho = orc_out_h(p), Wo = orc_out_w(p);
  const int K = p->kh * p->kw, M = 2 * p->groups * K;
  const long HoWo = (long)Ho * Wo;
  const long CK = (long)p->c_in * K;
  double *off = (double *)malloc(sizeof(double) * p->n * M * HoWo);
  double *col = (double *)malloc(sizeof(double) * p->n * CK * HoWo);
  if (!off || !col) {
    free(off);
    free(col);
    return ORC_NO_MEMORY;
  }
  orc_offsets(p, x, w_off, b_off, offset_add, off);
  orc_column(p, x, off, col);
#pragma omp parallel for collapse(2) schedule(static)
  for (int n = 0; n < p->n; ++n)
    for (int o = 0; o < p->c_out; ++o) {
      double *dst = y + ((long)n * p->c_out + o) * HoWo;
      for (long q = 0; q < HoWo; ++q) dst[q] = 0.0;
      for (long ck = 0; ck < CK; ++ck) {
        const double wv = w[(long)o * CK + ck];
        const double *src = col + ((long)n * CK + ck) * HoWo;
        for (long q = 0; q < HoWo; ++q) dst[q] += wv * src[q];
      }
    }
  if (offset_out) memcpy(offset_out, off, sizeof(double) * p->n * M * HoWo);
  free(off);
  free(col);
  return ORC_OK;
}

/* Backward pass: exact derivative of orc_forward for the loss sum(y * gy),
 * taking the offsets `off` (including b_off and offset_add) as saved by the
 * forward pass.
 *   gw[o, c, k]      = sum_{n, q} gy[n, o, q] * col[n, c, k, q]
 *   gcol[n, c, k, q] = sum_o w[o, c, k] * gy[n, o, q]
 *   goff[n, 2(gK+k), q]   = sum_{c in g} gcol * dS/dpy
 *   goff[n, 2(gK+k)+1, q] = sum_{c in g} gcol * dS/dpx
 *   gx = adjoint of the sampling applied to gcol
 *        + adjoint of the offset convolution applied to goff
 *   gw_off[m, c, i, j] = sum_{n, q} goff[n, m, q] * xbar[n, c, at tap (i, j)]
 *   gb_off[m]          = sum_{n, q} goff[n, m, q]
 * goff is the gradient with respect to offset_add.  gb_off and goff may be
 * NULL.  Every output is overwritten. */
int orc_backward(const orc_problem *p, const double *x, const double *w_off,
                 const double *w, const double *off, const double *gy,
                 double *gx, double *gw_off, double *gb_off, double *gw,
                 double *goff_out) {
  int rc = orc_check(p);
  if (rc) return rc;
  const int Ho = orc_out_h(p), Wo = orc_out_w(p);
  const int K = p->kh * p->kw, M = 2 * p->groups * K, Cg = p->c_in / p->groups;
  const long HW = (long)p->h * p->w, HoWo = (long)Ho * Wo;
  const long CK = (long)p->c_in * K;
  double *col = (double *)malloc(sizeof(double) * p->n * CK * HoWo);
  double *gcol = (double *)malloc(sizeof(double) * p->n * CK * HoWo);
  double *goff = (double *)malloc(sizeof(double) * p->n * M * HoWo);
  if (!col || !gcol || !goff) {
    free(col);
    free(gcol);
    free(goff);
    return ORC_NO_MEMORY;
  }
  orc_column(p, x, off, col);

  /* main convolution: weight gradient */
#pragma omp parallel for collapse(2) schedule(static)
  for (int o = 0; o < p->c_out; ++o)
    for (long ck = 0; ck < CK; ++ck) {
      double s = 0.0;
      for (int n = 0; n < p->n; ++n) {
        const double *g = gy + ((long)n * p->c_out + o) * HoWo;
        const double *cc = col + ((long)n * CK + ck) * HoWo;
        for (long q = 0; q < HoWo; ++q) s += g[q] * cc[q];
      }
      gw[(long)o * CK + ck] = s;
    }

  /* main convolution: gradient of the deformed map */
#pragma omp parallel for collapse(2) schedule(static)
  for (int n = 0; n < p->n; ++n)
    for (long ck = 0; ck < CK; ++ck) {
      double *dst = gcol + ((long)n * CK + ck) * HoWo;
      for (long q = 0; q < HoWo; ++q) dst[q] = 0.0;
      for (int o = 0; o < p->c_out; ++o) {
        const double wv = w[(long)o * CK + ck];
        const double *g = gy + ((long)n * p->c_out + o) * HoWo;
        for (long q = 0; q < HoWo; ++q) dst[q] += wv * g[q];
      }
    }

  /* sampling: gradient with respect to the offsets */
#pragma omp parallel for collapse(2) schedule(static)
  for (int n = 0; n < p->n; ++n)
    for (int g = 0; g < p->groups; ++g)
      for (int i = 0; i < p->kh; ++i)
        for (int j = 0; j < p->kw; ++j) {
          const int k = i * p->kw + j;
          double *gdy = goff + ((long)n * M + 2 * (g * K + k)) * HoWo;
          double *gdx = gdy + HoWo;
          for (int ho = 0; ho < Ho; ++ho)
            for (int wo = 0; wo < Wo; ++wo) {
              double py, px, cy, cx, sy = 0.0, sx = 0.0;
              if (orc_sample_point(p, off, n, g, i, j, ho, wo, &py, &px, &cy, &cx))
                for (int c = g * Cg; c < (g + 1) * Cg; ++c) {
                  const double *plane = x + ((long)n * p->c_in + c) * HW;
                  const double gc =
                      gcol[(((long)n * p->c_in + c) * K + k) * HoWo +
                           (long)ho * Wo + wo];
                  double dpy, dpx;
                  orc_bilinear_grad_cell(plane, p->h, p->w, py, px, cy, cx, &dpy,
                                         &dpx);
                  sy += gc * dpy;
                  sx += gc * dpx;
                }
              gdy[(long)ho * Wo + wo] = sy;
              gdx[(long)ho * Wo + wo] = sx;
            }
        }

  /* sampling: gradient with respect to x */
  orc_column_adjoint(p, off, gcol, gx);

  /* offset convolution: its input gradient, added into gx */
#pragma omp parallel for collapse(2) schedule(static)
  for (int n = 0; n < p->n; ++n)
    for (int c = 0; c < p->c_in; ++c) {
      double *plane = gx + ((long)n * p->c_in + c) * HW;
      for (int m = 0; m < M; ++m) {
        const double *g = goff + ((long)n * M + m) * HoWo;
        for (int i = 0; i < p->kh; ++i)
          for (int j = 0; j < p->kw; ++j) {
            const double wv =
                w_off[(((long)m * p->c_in + c) * p->kh + i) * p->kw + j];
            for (int ho = 0; ho < Ho; ++ho)
              for (int wo = 0; wo < Wo; ++wo) {
                long a = (long)ho * p->stride_h - p->pad_h + (long)i * p->dil_h;
                long b = (long)wo * p->stride_w - p->pad_w + (long)j * p->dil_w;
                if (a < 0 || a >= p->h || b < 0 || b >= p->w) continue;
                plane[a * p->w + b] += wv * g[(long)ho * Wo + wo];
              }
          }
      }
    }

  /* offset convolution: weight and bias gradients */
#pragma omp parallel for collapse(2) schedule(static)
  for (int m = 0; m < M; ++m)
    for (int c = 0; c < p->c_in; ++c)
      for (int i = 0; i < p->kh; ++i)
        for (int j = 0; j < p->kw; ++j) {
          double s = 0.0;
          for (int n = 0; n < p->n; ++n) {
            const double *plane = x + ((long)n * p->c_in + c) * HW;
            const double *g = goff + ((long)n * M + m) * HoWo;
            for (int ho = 0; ho < Ho; ++ho)
              for (int wo = 0; wo < Wo; ++wo) {
                long a = (long)ho * p->stride_h - p->pad_h + (long)i * p->dil_h;
                long b = (long)wo * p->stride_w - p->pad_w + (long)j * p->dil_w;
                s += g[(long)ho * Wo + wo] * orc_pixel(plane, p->h, p->w, a, b);
              }
          }
          gw_off[(((long)m * p->c_in + c) * p->kh + i) * p->kw + j] = s;
        }
  if (gb_off)
    for (int m = 0; m < M; ++m) {
      double s = 0.0;
      for (int n = 0; n < p->n; ++n)
        for (long q = 0; q < HoWo; ++q) s += goff[((long)n * M + m) * HoWo + q];
      gb_off[m] = s;
    }
  if (goff_out) memcpy(goff_out, goff, sizeof(double) * p->n * M * HoWo);
  free(col);
  free(gcol);
  free(goff);
  return ORC_OK;
}

#ifdef _OPENMP
#include <omp.h>
#endif

/* Number of host threads the parallel loops above use. */
int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
