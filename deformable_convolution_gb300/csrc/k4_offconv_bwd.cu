// K4 on CUDA cores: backward of the offset convolution ("Following a
// deformable layer through DefT", Step 1 of 5, on the explainer page "DefT:
// Boosting Scalability of Deformable Convolution Operations on GPUs": a small
// standard convolution over the same input) for float32 problems and for bf16
// problems with more offset channels than the tensor-core kernel
// (k4_offconv_bwd_tc.cu) takes.  With goff the completed gradient of its
// output (summed over all channels by K3):
//   grad_x[b][c](q + tap k) += sum_m goff[b][m][q] * w_off[m][c][k]
//   grad_w_off[m][c][k]     += sum_{b,q} goff[b][m][q] * xbar[b][c](q + tap k)
//   grad_b_off[m]           += sum_{b,q} goff[b][m][q]
// One CTA owns a band of output rows (as K1 and K3) and a slice of input
// channels; it stages the band's receptive field of its channels (no margin:
// the offset convolution reads only the regular grid), keeps the band's goff
// on chip, accumulates grad_x in a shared window and flushes it with one
// float atomic per element.
#include "dc_band.cuh"

namespace dc {
namespace {

using band::kThreads;
constexpr int kMaxPx = band::kBandPx;
constexpr size_t kSmemBudget = 100 * 1024;

struct Plan {
  int R, TW, tiles_w, tiles_h, npx;
  int ps;  // pixel stride of the fp32 goff array
  int cpc, nslices;
  int rows, cols, plane;  // staged window: the band's receptive field
  size_t off_halo, off_gx, off_goff, off_tab, off_w, smem;
};

// offset channels per pass of the input gradient (w_off staged per pass)
constexpr int kMc = 12;

// The largest band and channel slice that fit and still give the grid at
// least two CTAs per SM (each CTA's phases are latency chains; a grid below
// the SM count leaves SMs idle); if none does, the fitting plan with the most
// CTAs; if nothing fits, the smallest.
__host__ Plan make_plan(const Geom& g, dc_dtype dt) {
  constexpr long long kMinGrid = 2 * 152;
  const bool bf16 = dt == DC_BF16;
  Plan best{}, most{};
  long long most_grid = 0;
  for (int px = kMaxPx; px >= 32; px /= 2) {
    const band::Shape sh = band::make_shape(g, 0, px);
    for (int cpc = 32; cpc >= 16; cpc -= 16) {
      Plan p{};
      p.R = sh.R;
      p.TW = sh.TW;
      p.npx = sh.npx;
      p.ps = px + 8;
      p.tiles_w = sh.tiles_w;
      p.tiles_h = sh.tiles_h;
      p.rows = sh.rows;
      p.cols = sh.cols;
      p.plane = sh.plane;
      p.cpc = cpc;
      p.nslices = (g.c_in + cpc - 1) / cpc;
      size_t at = 0;
      p.off_halo = at;
      at += (size_t)(bf16 ? cpc / 2 : cpc) * p.plane * 4;
      p.off_gx = at;
      at += (size_t)cpc * p.plane * 4;
      p.off_tab = at;  // pixel table [ps] + tap offsets [K]
      at += (size_t)(p.ps + g.K) * 4;
      p.off_goff = at;
      at += (size_t)g.M * p.ps * 4;
      at = (at + 15) / 16 * 16;
      p.off_w = at;  // w_off of the slice for one pass: [cpc][K][kMc] fp32
      at += (size_t)cpc * g.K * kMc * 4;
      p.smem = at;
      if (best.smem == 0 || p.smem < best.smem) best = p;
      if (p.smem <= kSmemBudget) {
        const long long grid = (long long)p.nslices * p.tiles_w * p.tiles_h * g.n;
        if (grid >= kMinGrid) return p;
        if (grid > most_grid) {
          most = p;
          most_grid = grid;
        }
      }
    }
  }
  return most_grid > 0 ? most : best;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) k4_offconv_bwd(OffconvBwdArgs a, Plan pl) {
  extern __shared__ __align__(16) unsigned char smem[];
  const Geom g = a.g;
  const T* __restrict__ x = static_cast<const T*>(a.x);
  const T* __restrict__ w_off = static_cast<const T*>(a.w_off);
  const int slice = (int)(blockIdx.x % pl.nslices);
  const int tw_idx = (int)(blockIdx.x / pl.nslices);
  const int ho0 = blockIdx.y * pl.R, wo0 = tw_idx * pl.TW;
  const int n = blockIdx.z;
  const int c_begin = slice * pl.cpc;
  const int ncur = min(g.c_in, c_begin + pl.cpc) - c_begin;
  const int ylo = ho0 * g.sh - g.ph, xlo = wo0 * g.sw - g.pw;
  const int tid = threadIdx.x;
  const int PL = pl.plane, PS = pl.ps, npx = pl.npx, M = g.M;
  const long long img = (long long)n * g.c_in * g.hw;
  const int margin = 0;

  uint32_t* xw = reinterpret_cast<uint32_t*>(smem + pl.off_halo);
  float* gxs = reinterpret_cast<float*>(smem + pl.off_gx);     // [cpc][PL]
  int* pix = reinterpret_cast<int*>(smem + pl.off_tab);        // (row << 16 | col)
  int* tapoff = pix + PS;

  for (int k = tid; k < g.K; k += kThreads) {
    const int i = k / g.kw;
    tapoff[k] = i * g.dh * pl.cols + (k - i * g.kw) * g.dw;
  }
  band::stage_window<T>(x, g, img, c_begin, pl.cpc, ylo, xlo, pl.rows, pl.cols, PL, xw);
  for (int idx = tid; idx < pl.cpc * PL; idx += kThreads) gxs[idx] = 0.f;
  // the offset gradient is K3's output; grad_x / grad_w_off / grad_b_off were
  // cleared by the GCOL GEMM before K3 started
  pdl_wait();
  pdl_release();

  {
    float* goff = reinterpret_cast<float*>(smem + pl.off_goff);  // [M][PS]
    band::fill_pixel_table(pix, npx, pl.TW);
    __syncthreads();
    {
      band::Walk2 w;
      w.init(tid, kThreads, npx);
      while (w.a < M) {
        const int m = w.a, px = w.b;
        w.next();
        const int e = pix[px];
        const int ho = ho0 + (e >> 16), wo = wo0 + (e & 0xffff);
        float v = 0.f;
        if (ho < g.ho && wo < g.wo)
          v = a.goff[((long long)n * M + m) * g.howo + (long long)ho * g.wo + wo];
        goff[m * PS + px] = v;
      }
    }
    __syncthreads();
    // ---------------------------------------------------------------- offset-conv input gradient
    // for each (channel, pixel): sum over offset channels of goff * w_off at every
    // tap, added to the window position that tap reads; per pass of kMc offset
    // channels the slice's w_off is staged as [channel][tap][m] (zeros past M
    // and past the last channel), so the kMc-term sums add in the same order
    {
      float* wsm = reinterpret_cast<float*>(smem + pl.off_w);
      const int wn = pl.cpc * g.K * kMc;
      for (int m0 = 0; m0 < M; m0 += kMc) {
        __syncthreads();  // the previous pass is done with wsm
        for (int idx = tid; idx < wn; idx += kThreads) {
          const int cl = idx / (g.K * kMc), r = idx - cl * (g.K * kMc);
          const int k = r / kMc, t = r - k * kMc;
          wsm[idx] = (cl < ncur && m0 + t < M)
                         ? ld_f(w_off + ((long long)(m0 + t) * g.c_in + c_begin + cl) * g.K + k)
                         : 0.f;
        }
        __syncthreads();
        band::Walk2 w;
        w.init(tid, kThreads, npx);
        while (w.a < ncur) {
          const int cl = w.a, px = w.b;
          w.next();
          const int e = pix[px];
          const int pos = ((e >> 16) * g.sh + margin) * pl.cols + (e & 0xffff) * g.sw + margin;
          float* gp = gxs + cl * PL + pos;
          float gv[kMc];
  #pragma unroll
          for (int t = 0; t < kMc; ++t) gv[t] = (m0 + t < M) ? goff[(m0 + t) * PS + px] : 0.f;
          const float* wk = wsm + cl * g.K * kMc;
          for (int k = 0; k < g.K; ++k) {
            float s = 0.f;
  #pragma unroll
            for (int t = 0; t < kMc; ++t)
              if (m0 + t < M) s = __fmaf_rn(gv[t], wk[k * kMc + t], s);
            if (s != 0.f) atomicAdd(gp + tapoff[k], s);
          }
        }
      }
    }

    // ---------------------------------------------------------------- offset-conv weight gradient
    {
      constexpr int kMw = 12;
      const int nmc = (M + kMw - 1) / kMw;
      band::Walk3 w;
      w.init(tid, kThreads, g.K, nmc);
      while (w.a < ncur) {
        const int cl = w.a, k = w.b, m0 = w.c * kMw;
        w.next();
        float acc[kMw];
  #pragma unroll
        for (int t = 0; t < kMw; ++t) acc[t] = 0.f;
        const int toff = tapoff[k] + margin * pl.cols + margin;
        for (int px = 0; px < npx; ++px) {
          const int e = pix[px];
          const float xv = band::staged<T>(xw, PL, cl, (e >> 16) * g.sh * pl.cols + (e & 0xffff) * g.sw + toff);
  #pragma unroll
          for (int t = 0; t < kMw; ++t)
            if (m0 + t < M) acc[t] = __fmaf_rn(goff[(m0 + t) * PS + px], xv, acc[t]);
        }
        float* dst = a.gw_off + (long long)(c_begin + cl) * g.K + k;
  #pragma unroll
        for (int t = 0; t < kMw; ++t)
          if (m0 + t < M) atomicAdd(dst + (long long)(m0 + t) * g.c_in * g.K, acc[t]);
      }
    }
    if (a.gb_off && slice == 0) {
      for (int m = tid; m < M; m += kThreads) {
        float s = 0.f;
        for (int px = 0; px < npx; ++px) s += goff[m * PS + px];
        atomicAdd(a.gb_off + m, s);
      }
    }
  }
  __syncthreads();

  // flush the grad_x window (neighbouring bands' windows overlap)
  {
    band::Walk3 w;
    w.init(tid, kThreads, pl.rows, pl.cols);
    while (w.a < ncur) {
      const int cl = w.a, r = w.b, q = w.c;
      w.next();
      const int yy = ylo + r, xx = xlo + q;
      if (yy < 0 || yy >= g.h || xx < 0 || xx >= g.w) continue;
      const float v = gxs[cl * PL + r * pl.cols + q];
      if (v != 0.f) atomicAdd(a.gx + img + (long long)(c_begin + cl) * g.hw + (long long)yy * g.w + xx, v);
    }
  }
}

template <typename T>
cudaError_t launch_t(const OffconvBwdArgs& a, const Plan& pl, cudaStream_t s) {
  auto kern = k4_offconv_bwd<T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pl.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(pl.nslices * pl.tiles_w), (unsigned)pl.tiles_h, (unsigned)a.g.n);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a, pl);
  note_launches(1);
  return e;
}

}  // namespace

size_t offconv_bwd_smem_bytes(const Geom& g, dc_dtype dt) {
  return offconv_bwd_tc_supported(g, dt) ? offconv_bwd_tc_smem_bytes(g) : make_plan(g, dt).smem;
}

cudaError_t launch_offconv_bwd(const OffconvBwdArgs& a, dc_dtype dt, cudaStream_t s) {
  if (offconv_bwd_tc_supported(a.g, dt)) return launch_offconv_bwd_tc(a, s);
  const Plan pl = make_plan(a.g, dt);
  return dt == DC_BF16 ? launch_t<__nv_bfloat16>(a, pl, s) : launch_t<float>(a, pl, s);
}

}  // namespace dc
