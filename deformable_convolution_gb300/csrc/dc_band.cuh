// Band tiling shared by the fused forward kernel (K1) and the fused backward
// kernel (K3).
//
// The explainer page "DefT: Boosting Scalability of Deformable Convolution
// Operations on GPUs" tiles by the output's spatial dimensions and pads each
// tile's input window by a margin sized to the offset distribution ("Why it
// works", "The idea").  Here a tile is a band of R full-width output rows
// (at most kBandPx pixels); its input window is the band's receptive field plus
// `margin` pixels on each side.  Channels are split into slices of CPC, one
// slice per CTA of a thread-block cluster.
#pragma once

#include "dc_common.cuh"

namespace dc {
namespace band {

constexpr int kThreads = 256;  // block size of K3 and K4 (the helpers take any)
constexpr int kBandPx = 128;  // largest band; smaller ones are tried when shared memory is short
constexpr int kMaxCluster = 8;

struct Shape {
  int R, TW, tiles_w, tiles_h, npx;
  int in_rows, in_cols;  // receptive field of the band
  int rows, cols;        // staged window (receptive field + 2 * margin)
  int plane;             // padded 32-bit words per staged plane
};

// Words per plane, rounded so that consecutive planes start 8 banks apart.
__host__ inline int pad_plane(int v) {
  int p = (v + 31) / 32 * 32 + 8;
  if (p - 32 >= v) p -= 32;
  return p;
}

// Tile of R output rows x TW output columns and its staged input window.
__host__ inline Shape shape_rt(const Geom& g, int margin, int R, int TW) {
  Shape s{};
  s.TW = TW;
  s.R = R;
  s.npx = s.R * s.TW;
  s.tiles_w = (int)ceil_div_ll(g.wo, s.TW);
  s.tiles_h = (int)ceil_div_ll(g.ho, s.R);
  s.in_rows = (s.R - 1) * g.sh + (g.kh - 1) * g.dh + 1;
  s.in_cols = (s.TW - 1) * g.sw + (g.kw - 1) * g.dw + 1;
  s.rows = s.in_rows + 2 * margin;
  s.cols = s.in_cols + 2 * margin;
  s.plane = pad_plane(s.rows * s.cols);
  return s;
}

// Per-shape cost model for the tile of at most `px` output pixels (the
// page's tiling by output spatial dimensions, "The idea", with tile sizes left
// open there).  Candidates: full-width rows (TW = Wo when Wo <= px) and 2-D
// tiles of TW = 8, 16, ... columns.  Each is scored by the input positions all
// tiles stage -- receptive field plus margin, the work of staging, clearing
// and flushing the windows -- plus a fixed cost per tile (tables, weights,
// barriers); full-width rows get a bonus for the contiguous row runs the
// vector paths use, 8-column tiles a penalty for their half-sector writes of
// the deformed map, and ties go to the wider tile.  Wide, dilated layers thus
// get square-ish tiles instead of one-row bands whose window is mostly halo.
constexpr double kTileFixedPositions = 512.0;
constexpr double kFullWidthBonus = 0.85;
constexpr double kNarrowPenalty = 1.15;

__host__ inline Shape make_shape(const Geom& g, int margin, int px) {
  Shape best{};
  double best_cost = 0.0;
  auto consider = [&](int TW) {
    int R = px / TW;
    if (R < 1) return;
    if (R > g.ho) R = g.ho;
    R = (int)ceil_div_ll(g.ho, ceil_div_ll(g.ho, R));  // same tile count, rows balanced
    const Shape s = shape_rt(g, margin, R, TW);
    double cost = (double)s.tiles_w * s.tiles_h * ((double)s.rows * s.cols + kTileFixedPositions);
    if (TW == g.wo) cost *= kFullWidthBonus;
    else if (TW < 16) cost *= kNarrowPenalty;
    if (best.npx == 0 || cost <= best_cost) {
      best = s;
      best_cost = cost;
    }
  };
  if (g.wo <= px) consider(g.wo);
  for (int tw = 8; tw <= px; tw *= 2)
    if (tw < g.wo) consider(tw);
  if (best.npx == 0) consider(px < g.wo ? px : g.wo);
  return best;
}

// Per (pixel, tap, group) sampling state.
struct Tap {
  bool inside, fast;
  float ly, lx;
  int y0, x0;  // lower corner, image coordinates
};

__device__ __forceinline__ Tap make_tap(float py, float pxf, const Geom& g, int ylo, int xlo,
                                        int rows, int cols) {
  Tap t;
  t.inside = touches_image(py, pxf, g.h, g.w);
  t.fast = false;
  t.ly = t.lx = 0.f;
  t.y0 = t.x0 = 0;
  if (t.inside) {
    const float fy = floorf(py), fx = floorf(pxf);
    t.ly = py - fy;
    t.lx = pxf - fx;
    t.y0 = (int)fy;
    t.x0 = (int)fx;
    const int ry = t.y0 - ylo, rx = t.x0 - xlo;
    t.fast = ry >= 0 && ry + 1 < rows && rx >= 0 && rx + 1 < cols;
  }
  return t;
}

template <typename T>
__device__ __forceinline__ float gload(const T* plane, const Geom& g, int y, int x) {
  return (y >= 0 && y < g.h && x >= 0 && x < g.w) ? ld_f(plane + (long long)y * g.w + x) : 0.0f;
}

__device__ __forceinline__ uint32_t bf16_bits(const __nv_bfloat16* p) {
  return (uint32_t)(*reinterpret_cast<const unsigned short*>(p));
}

__device__ __forceinline__ uint32_t raw_bits(const __nv_bfloat16* p) { return bf16_bits(p); }
__device__ __forceinline__ uint32_t raw_bits(const float* p) { return __float_as_uint(*p); }

// Walks the flattened index of a [A x B] grid in steps of `step` without
// divisions after the first element (step is split once into step = da*B + db).
struct Walk2 {
  int a, b, da, db, B;
  __device__ __forceinline__ void init(int start, int step, int nb) {
    B = nb;
    a = start / nb;
    b = start - a * nb;
    da = step / nb;
    db = step - da * nb;
  }
  __device__ __forceinline__ void next() {
    b += db;
    a += da;
    if (b >= B) {
      b -= B;
      a += 1;
    }
  }
};

// Same for a [A x B x C] grid.
struct Walk3 {
  int a, b, c, da, db, dc, B, C;
  __device__ __forceinline__ void init(int start, int step, int nb, int nc) {
    B = nb;
    C = nc;
    const int bc = nb * nc;
    a = start / bc;
    int r = start - a * bc;
    b = r / nc;
    c = r - b * nc;
    da = step / bc;
    r = step - da * bc;
    db = r / nc;
    dc = r - db * nc;
  }
  __device__ __forceinline__ void next() {
    c += dc;
    b += db;
    a += da;
    if (c >= C) {
      c -= C;
      b += 1;
    }
    if (b >= B) {
      b -= B;
      a += 1;
    }
  }
};

// Stages the window [ylo, ylo+rows) x [xlo, xlo+cols) of channels
// [c_begin, c_begin + cpc) of image `img` into shared memory, zero outside the
// image and beyond c_in.  bf16: one 32-bit word per pixel per channel pair
// (low half = even channel); fp32: one word per pixel per channel.  Plane u
// starts at dst + u * plane.  Each thread keeps kBatch independent global loads
// in flight; lanes run along window rows, so loads are coalesced.
// Fast path of stage_window for bf16 when image rows are whole 8-byte
// quads (W % 4 == 0, 8-byte aligned planes): a task is (channel pair, window
// row, aligned 4-pixel quad of the image row); it reads one 8-byte quad of each
// of the two channels and writes up to four pair words.  Quads lie either
// wholly inside or wholly outside the image, so no load straddles an edge.
__device__ __forceinline__ void stage_window_quads(const __nv_bfloat16* __restrict__ x,
                                                   const Geom& g, long long img, int c_begin,
                                                   int cpc, int ylo, int xlo, int rows, int cols,
                                                   int plane, uint32_t* dst) {
  constexpr int kBatch = 4;
  const int q_lo = (xlo >= 0 ? xlo : xlo - 3) / 4;  // floor(xlo / 4)
  const int q_hi = (xlo + cols - 1 >= 0 ? xlo + cols - 1 : xlo + cols - 4) / 4;
  const int nq = q_hi - q_lo + 1;
  const int units = cpc / 2;
  Walk3 w;
  w.init(threadIdx.x, blockDim.x, rows, nq);
  while (w.a < units) {
    uint2 v0[kBatch], v1[kBatch];
    int uu[kBatch], rr[kBatch], qq[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      v0[j] = v1[j] = make_uint2(0u, 0u);
      uu[j] = -1;
      if (w.a < units) {
        uu[j] = w.a;
        rr[j] = w.b;
        qq[j] = q_lo + w.c;
        const int yy = ylo + w.b, x0 = 4 * qq[j];
        if (yy >= 0 && yy < g.h && x0 >= 0 && x0 < g.w) {
          const int c0 = c_begin + 2 * w.a;
          const __nv_bfloat16* p = x + img + (long long)c0 * g.hw + (long long)yy * g.w + x0;
          if (c0 < g.c_in) v0[j] = *reinterpret_cast<const uint2*>(p);
          if (c0 + 1 < g.c_in) v1[j] = *reinterpret_cast<const uint2*>(p + g.hw);
        }
        w.next();
      }
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      if (uu[j] < 0) continue;
      // pixel i of the quad: low half = channel c0, high half = channel c0 + 1
      const uint32_t pw[4] = {__byte_perm(v0[j].x, v1[j].x, 0x5410), __byte_perm(v0[j].x, v1[j].x, 0x7632),
                              __byte_perm(v0[j].y, v1[j].y, 0x5410), __byte_perm(v0[j].y, v1[j].y, 0x7632)};
      uint32_t* row = dst + uu[j] * plane + rr[j] * cols;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int col = 4 * qq[j] + i - xlo;
        if (col >= 0 && col < cols) row[col] = pw[i];
      }
    }
  }
}

template <typename T>
__device__ __forceinline__ void stage_window(const T* __restrict__ x, const Geom& g,
                                             long long img, int c_begin, int cpc, int ylo,
                                             int xlo, int rows, int cols, int plane,
                                             uint32_t* dst) {
  constexpr bool kPairs = sizeof(T) == 2;
  if (kPairs && (g.w & 3) == 0 && (cpc & 1) == 0 &&
      (reinterpret_cast<uintptr_t>(x) & 7) == 0) {
    stage_window_quads(reinterpret_cast<const __nv_bfloat16*>(x), g, img, c_begin, cpc, ylo, xlo,
                       rows, cols, plane, dst);
    return;
  }
  constexpr int kBatch = 16;
  const int units = kPairs ? cpc / 2 : cpc;
  Walk3 w;
  w.init(threadIdx.x, blockDim.x, rows, cols);
  while (w.a < units) {
    uint32_t v[kBatch];
    int at[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      v[j] = 0u;
      at[j] = -1;
      if (w.a < units) {
        const int u = w.a;
        at[j] = u * plane + w.b * cols + w.c;
        const int yy = ylo + w.b, xx = xlo + w.c;
        if (yy >= 0 && yy < g.h && xx >= 0 && xx < g.w) {
          const long long pix = (long long)yy * g.w + xx;
          if (kPairs) {
            const int c0 = c_begin + 2 * u;
            if (c0 < g.c_in) v[j] = raw_bits(x + img + (long long)c0 * g.hw + pix);
            if (c0 + 1 < g.c_in) v[j] |= raw_bits(x + img + (long long)(c0 + 1) * g.hw + pix) << 16;
          } else {
            const int c = c_begin + u;
            if (c < g.c_in) v[j] = raw_bits(x + img + (long long)c * g.hw + pix);
          }
        }
        w.next();
      }
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      if (at[j] >= 0) dst[at[j]] = v[j];
  }
}

// Per-band table of output pixels: packs (row in band, column in band) into
// one int so inner loops need no division by the band width.
__device__ __forceinline__ void fill_pixel_table(int* tab, int npx, int TW) {
  for (int px = threadIdx.x; px < npx; px += blockDim.x) {
    const int r = px / TW;
    tab[px] = (r << 16) | (px - r * TW);
  }
}

// Value of channel `cl` (relative to the slice) at staged word offset `pos`.
template <typename T>
__device__ __forceinline__ float staged(const uint32_t* xs, int plane, int cl, int pos) {
  if (sizeof(T) == 2) {
    const uint32_t w = xs[(cl >> 1) * plane + pos];
    return __uint_as_float(((cl & 1) ? w : (w << 16)) & 0xffff0000u);
  }
  return __uint_as_float(xs[cl * plane + pos]);
}

}  // namespace band
}  // namespace dc
