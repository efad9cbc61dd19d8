// Host-side checks of the tensor-core offset-convolution backward's plan and
// of the accumulator-order layout of its grad_w_off partials, over a sweep of
// layer geometries (compiled and run by tests/test_host_layout.py; no GPU).
//
//  * the partials' order maps every (offset channel, input channel, tap) of
//    grad_w_off [M][C_in][K] from exactly one element, and only padding
//    elements map nowhere;
//  * the input window is wide enough for the receptive field shifted by the
//    even-column alignment, has an even width, and every window position a
//    pixel's tap reads lies inside the staged plane;
//  * the padded sizes the kernel's loops assume hold (pixels to 16, window
//    positions to 8, offset channels to 8 and 16) and shared memory fits.
#include "../../deformable_convolution_gb300/csrc/k4_offconv_bwd_tc.cu"

#include <cstdio>
#include <vector>

namespace dc {
void note_launches(unsigned) {}
}  // namespace dc

using namespace dc;

static int failures = 0;
#define CHECK(cond, ...)                  \
  do {                                    \
    if (!(cond)) {                        \
      if (failures < 20) {                \
        printf("FAIL %s: ", #cond);       \
        printf(__VA_ARGS__);              \
        printf("\n");                     \
      }                                   \
      ++failures;                         \
    }                                     \
  } while (0)

static bool make_geom(Geom& g, int n, int c, int h, int w, int k, int s, int p, int d, int gr) {
  g = Geom{};
  g.n = n; g.c_in = c; g.h = h; g.w = w; g.c_out = 8;
  g.kh = g.kw = k; g.sh = g.sw = s; g.ph = g.pw = p; g.dh = g.dw = d; g.groups = gr;
  g.ho = (h + 2 * p - d * (k - 1) - 1) / s + 1;
  g.wo = (w + 2 * p - d * (k - 1) - 1) / s + 1;
  if (g.ho < 1 || g.wo < 1 || c % gr) return false;
  g.K = k * k; g.M = 2 * gr * g.K; g.cg = c / gr; g.kdim = c * g.K;
  g.hw = (long long)h * w; g.howo = (long long)g.ho * g.wo;
  return offconv_bwd_tc_supported(g, DC_BF16);
}

static void check_partials(const Geom& g, const char* tag) {
  const long long count = gwo_frag_count(g.M, g.c_in, g.K);
  const long long target = (long long)g.M * g.c_in * g.K;
  CHECK(count % 128 == 0 && count >= target, "%s count %lld target %lld", tag, count, target);
  std::vector<int> hits((size_t)target, 0);
  long long valid = 0;
  for (long long e4 = 0; e4 < count / 4; ++e4) {
    long long d[4];
    gwo_frag_dest4((int)e4, g.M, g.c_in, g.K, d);
    for (int h = 0; h < 4; ++h) {
      const long long e = 4 * e4 + h;
      // decode the order independently: [slice][tap][m tile][lane][4]
      const int lane = (int)((e >> 2) & 31), mtiles = (g.M + 7) / 8;
      const long long r = e >> 7;
      const int mt = (int)(r % mtiles), k = (int)((r / mtiles) % g.K), slice = (int)(r / mtiles / g.K);
      const int m = mt * 8 + 2 * (lane & 3) + (h & 1), c = slice * 16 + (lane >> 2) + 8 * (h >> 1);
      const bool pad = m >= g.M || c >= g.c_in;
      CHECK(pad == (d[h] < 0), "%s e=%lld pad=%d d=%lld", tag, e, (int)pad, d[h]);
      if (d[h] >= 0) {
        CHECK(d[h] == ((long long)m * g.c_in + c) * g.K + k, "%s e=%lld d=%lld", tag, e, d[h]);
        CHECK(d[h] < target, "%s e=%lld d=%lld out of range", tag, e, d[h]);
        if (d[h] < target) ++hits[(size_t)d[h]];
        ++valid;
      }
    }
  }
  CHECK(valid == target, "%s valid %lld target %lld", tag, valid, target);
  for (long long i = 0; i < target; ++i) CHECK(hits[(size_t)i] == 1, "%s element %lld hit %d times", tag, i, hits[(size_t)i]);
}

static void check_plan(const Geom& g, const char* tag) {
  const TcPlan p = pick_tc_plan(g);
  const int in_cols = (p.TW - 1) * g.sw + (g.kw - 1) * g.dw + 1;
  const int in_rows = (p.R - 1) * g.sh + (g.kh - 1) * g.dh + 1;
  CHECK((p.cols & 1) == 0, "%s cols %d odd", tag, p.cols);
  CHECK(p.cols >= in_cols + 1, "%s cols %d receptive field %d", tag, p.cols, in_cols);
  CHECK(p.rows >= in_rows, "%s rows %d receptive field %d", tag, p.rows, in_rows);
  CHECK(p.npos == p.rows * p.cols, "%s npos %d rows*cols %d", tag, p.npos, p.rows * p.cols);
  CHECK(p.nq % 8 == 0 && p.nq >= p.npos && p.nq < p.npos + 8, "%s nq %d", tag, p.nq);
  CHECK(p.xplane >= p.npos, "%s xplane %d npos %d", tag, p.xplane, p.npos);
  CHECK(p.pxp % 16 == 0 && p.pxp >= p.npx && p.npx == p.R * p.TW, "%s pxp %d npx %d", tag, p.pxp, p.npx);
  CHECK(p.mp8 % 8 == 0 && p.mp8 >= g.M && p.mp16 % 16 == 0 && p.mp16 >= g.M, "%s mp8/16", tag);
  CHECK(p.smem <= 227 * 1024, "%s smem %zu", tag, p.smem);
  CHECK((long long)p.tiles_w * p.TW >= g.wo && (long long)p.tiles_h * p.R >= g.ho, "%s tiles", tag);
  // every window position a pixel's tap reads, for either column shift
  for (int xs = 0; xs < 2; ++xs)
    for (int px = 0; px < p.npx; ++px)
      for (int i = 0; i < g.kh; ++i)
        for (int j = 0; j < g.kw; ++j) {
          const int r = px / p.TW, c = px % p.TW;
          const int q = (r * g.sh + i * g.dh) * p.cols + c * g.sw + j * g.dw + xs;
          CHECK(q >= 0 && q < p.npos && (c * g.sw + j * g.dw + xs) < p.cols, "%s px %d tap %d,%d xs %d q %d",
                tag, px, i, j, xs, q);
        }
}

int main() {
  const int cs[] = {1, 3, 8, 16, 17, 40, 64, 128, 256};
  const int hs[] = {1, 5, 9, 28, 50, 56};
  const int ws[] = {1, 4, 9, 28, 84, 112, 130};
  const int ks[] = {1, 2, 3, 5};
  int cases = 0;
  for (int c : cs)
    for (int h : hs)
      for (int w : ws)
        for (int k : ks)
          for (int s = 1; s <= 2; ++s)
            for (int p = 0; p <= 2; ++p)
              for (int d = 1; d <= 2; ++d)
                for (int gr : {1, 2, 4}) {
                  Geom g;
                  if (!make_geom(g, 2, c, h, w, k, s, p, d, gr)) continue;
                  char tag[128];
                  snprintf(tag, sizeof tag, "c%d h%d w%d k%d s%d p%d d%d g%d", c, h, w, k, s, p, d, gr);
                  check_plan(g, tag);
                  if (h == 9 && (w == 9 || w == 130) && p == 1) check_partials(g, tag);
                  ++cases;
                }
  // the benchmark layers
  Geom g;
  if (make_geom(g, 8, 128, 28, 28, 3, 1, 1, 1, 1)) { check_plan(g, "res3"); check_partials(g, "res3"); ++cases; }
  if (make_geom(g, 2, 256, 50, 84, 3, 1, 1, 1, 1)) { check_plan(g, "res4"); check_partials(g, "res4"); ++cases; }
  if (make_geom(g, 16, 64, 112, 112, 3, 1, 2, 2, 4)) { check_plan(g, "early"); check_partials(g, "early"); ++cases; }
  printf("%d geometries, %d failures\n", cases, failures);
  return failures == 0 && cases > 100 ? 0 : 1;
}
