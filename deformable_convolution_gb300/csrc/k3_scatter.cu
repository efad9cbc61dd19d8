// K3: backward of the bilinear sampling step.
//
// For each sampling point (image b, offset group g, tap k, output pixel q) and
// each channel c of the group, with gc = gcol[c*K + k][b][q]:
//   grad_x[b][c] at the four corners += corner weight * gc      (inside image)
//   grad_dy += gc * ((1-lx) (v10 - v00) + lx (v11 - v01))
//   grad_dx += gc * ((1-ly) (v01 - v00) + ly (v11 - v10))
// which is the exact derivative of the four-neighbour blend ("The argument in
// one glance / Why it fell short" on the explainer page "DefT: Boosting
// Scalability of Deformable Convolution Operations on GPUs"), with the lower
// corner at floor(p) so integer coordinates take the right-sided difference.
//
// Threads run along output pixels, so gcol reads and offset reads/writes are
// coalesced and each offset-gradient sum stays in one thread's registers.
// grad_x is scattered with fp32 atomics; lanes whose corner addresses coincide
// are merged inside the warp first (warp-aggregated atomics), which removes
// most of the traffic when offsets pull neighbouring taps onto one pixel.
#include "dc_common.cuh"

namespace dc {
namespace {

constexpr int kThreads = 256;

// Adds v to *addr, one atomic per distinct address among the active lanes:
// lanes with equal addresses are summed in lane order by their lowest lane.
__device__ __forceinline__ void warp_aggregated_add(float* addr, float v, bool active) {
  const unsigned mask = __ballot_sync(0xffffffffu, active);
  if (!active) return;
  const unsigned peers = __match_any_sync(mask, reinterpret_cast<unsigned long long>(addr));
  const int leader = __ffs(peers) - 1;
  float total = 0.0f;
  for (unsigned rest = peers; rest; rest &= rest - 1)
    total += __shfl_sync(peers, v, __ffs(rest) - 1);
  if ((int)(threadIdx.x & 31) == leader) atomicAdd(addr, total);
}

template <typename T>
__global__ void __launch_bounds__(kThreads) k3_scatter(ScatterArgs a) {
  const Geom g = a.g;
  const T* __restrict__ x = static_cast<const T*>(a.x);
  const long long howo = g.howo;
  const long long total = (long long)g.n * g.groups * g.K * howo;
  // one warp-uniform loop so that every lane reaches the warp collectives
  for (long long base = (long long)blockIdx.x * kThreads; base < total;
       base += (long long)gridDim.x * kThreads) {
    const long long idx = base + threadIdx.x;
    const bool live = idx < total;
    long long q = 0;
    int k = 0, gg = 0, b = 0;
    if (live) {
      q = idx % howo;
      long long t = idx / howo;
      k = (int)(t % g.K);
      t /= g.K;
      gg = (int)(t % g.groups);
      b = (int)(t / g.groups);
    }
    const int ho = (int)(q / g.wo), wo = (int)(q % g.wo);
    const int i = k / g.kw, j = k % g.kw;
    float py = 0.f, pxf = 0.f;
    const long long off_dy = ((long long)b * g.M + 2 * (gg * g.K + k)) * howo + q;
    if (live) {
      py = (float)(ho * g.sh - g.ph + i * g.dh) + a.off[off_dy];
      pxf = (float)(wo * g.sw - g.pw + j * g.dw) + a.off[off_dy + howo];
    }
    const bool inside = live && touches_image(py, pxf, g.h, g.w);
    float ly = 0.f, lx = 0.f;
    int y0 = 0, x0 = 0;
    if (inside) {
      const float fy = floorf(py), fx = floorf(pxf);
      ly = py - fy;
      lx = pxf - fx;
      y0 = (int)fy;
      x0 = (int)fx;
    }
    const bool r0 = inside && y0 >= 0 && y0 < g.h, r1 = inside && y0 + 1 < g.h && y0 + 1 >= 0;
    const bool c0 = inside && x0 >= 0 && x0 < g.w, c1 = inside && x0 + 1 < g.w && x0 + 1 >= 0;
    const float hy = 1.0f - ly, hx = 1.0f - lx;
    const float w00 = hy * hx, w01 = hy * lx, w10 = ly * hx, w11 = ly * lx;
    float sdy = 0.f, sdx = 0.f;
    for (int cl = 0; cl < g.cg; ++cl) {
      const int c = gg * g.cg + cl;
      float gc = 0.f;
      if (inside) gc = a.gcol[(long long)(c * g.K + k) * a.gcol_layout.row + (long long)b * a.gcol_layout.img + q];
      const long long plane = ((long long)b * g.c_in + c) * g.hw;
      float v00 = 0.f, v01 = 0.f, v10 = 0.f, v11 = 0.f;
      if (r0 && c0) v00 = ld_f(x + plane + (long long)y0 * g.w + x0);
      if (r0 && c1) v01 = ld_f(x + plane + (long long)y0 * g.w + x0 + 1);
      if (r1 && c0) v10 = ld_f(x + plane + (long long)(y0 + 1) * g.w + x0);
      if (r1 && c1) v11 = ld_f(x + plane + (long long)(y0 + 1) * g.w + x0 + 1);
      sdy = __fmaf_rn(gc, hx * (v10 - v00) + lx * (v11 - v01), sdy);
      sdx = __fmaf_rn(gc, hy * (v01 - v00) + ly * (v11 - v10), sdx);
      float* gx = a.gx + plane;
      warp_aggregated_add(gx + (long long)y0 * g.w + x0, w00 * gc, r0 && c0);
      warp_aggregated_add(gx + (long long)y0 * g.w + x0 + 1, w01 * gc, r0 && c1);
      warp_aggregated_add(gx + (long long)(y0 + 1) * g.w + x0, w10 * gc, r1 && c0);
      warp_aggregated_add(gx + (long long)(y0 + 1) * g.w + x0 + 1, w11 * gc, r1 && c1);
    }
    if (live) {
      a.goff[off_dy] = sdy;
      a.goff[off_dy + howo] = sdx;
    }
  }
}

}  // namespace

cudaError_t launch_scatter(const ScatterArgs& a, dc_dtype dt, cudaStream_t s) {
  const Geom& g = a.g;
  const long long total = (long long)g.n * g.groups * g.K * g.howo;
  if (total == 0) return cudaSuccess;
  long long blocks = ceil_div_ll(total, kThreads);
  if (blocks > 152LL * 16) blocks = 152LL * 16;
  if (dt == DC_BF16)
    k3_scatter<__nv_bfloat16><<<(unsigned)blocks, kThreads, 0, s>>>(a);
  else
    k3_scatter<float><<<(unsigned)blocks, kThreads, 0, s>>>(a);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace dc
