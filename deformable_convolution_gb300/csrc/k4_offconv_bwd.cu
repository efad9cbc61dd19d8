// K4: backward of the offset convolution ("Following a deformable layer
// through DefT", Step 1 of 5, on the explainer page "DefT: Boosting
// Scalability of Deformable Convolution Operations on GPUs": a small standard
// convolution over the same input).  With goff the completed gradient of its
// output (summed over all channels by K3):
//   grad_x[b][c](q + tap k) += sum_m goff[b][m][q] * w_off[m][c][k]
//   grad_w_off[m][c][k]     += sum_{b,q} goff[b][m][q] * xbar[b][c](q + tap k)
//   grad_b_off[m]           += sum_{b,q} goff[b][m][q]
// One CTA owns a band of output rows (as K1 and K3) and a slice of input
// channels; it stages the band's receptive field of its channels (no margin:
// the offset convolution reads only the regular grid), keeps the band's goff
// on chip, runs both small contractions on tensor cores (bf16, fp32
// accumulation; CUDA cores for float32 problems or more than 80 offset
// channels), accumulates grad_x in a shared window and flushes it with one
// float atomic per element.
#include "dc_band.cuh"

namespace dc {
namespace {

using band::kThreads;
constexpr int kMaxPx = band::kBandPx;
constexpr size_t kSmemBudget = 100 * 1024;

struct Plan {
  int R, TW, tiles_w, tiles_h, npx;
  int ps;  // pixel stride of the fp32 goff array (CUDA-core path)
  int cpc, nslices;
  int rows, cols, plane;  // staged window: the band's receptive field
  // tensor path operand buffers (32-bit words of bf16 pairs)
  int mp16, pxp, nkp;     // M and pixels rounded up to 16, wA rows (K x cpc)
  int sa, sb, sw;         // word strides of gA [m][px/2], gB [px][m/2], wA [(k,c)][m/2]
  size_t off_halo, off_gx, off_goff, off_tab, off_ga, off_gb, off_wa, smem;
};

constexpr int kOffconvMmaMaxM = 80;

__host__ Plan make_plan(const Geom& g, dc_dtype dt) {
  const bool bf16 = dt == DC_BF16;
  const bool tensor = bf16 && g.M <= kOffconvMmaMaxM;
  Plan best{};
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
      p.mp16 = (g.M + 15) / 16 * 16;
      p.pxp = (p.npx + 15) / 16 * 16;
      p.nkp = g.K * cpc;  // wA rows (tap, channel), channels padded to cpc (a multiple of 16)
      p.sa = p.pxp / 2 + 4;  // rows 4 banks apart: conflict-free fragment loads
      p.sb = p.mp16 / 2 + 4;
      p.sw = p.mp16 / 2 + 4;
      size_t at = 0;
      p.off_halo = at;
      at += (size_t)(bf16 ? cpc / 2 : cpc) * p.plane * 4;
      p.off_gx = at;
      at += (size_t)cpc * p.plane * 4;
      p.off_tab = at;  // pixel table / positions [pxp or ps] + tap offsets [K]
      at += (size_t)((p.pxp > p.ps ? p.pxp : p.ps) + g.K) * 4;
      if (tensor) {
        p.off_ga = at;
        at += (size_t)p.mp16 * p.sa * 4;
        p.off_gb = at;
        at += (size_t)p.pxp * p.sb * 4;
        p.off_wa = at;  // also stages the band's fp32 goff [M][pxp] first
        {
          const size_t wa = (size_t)p.nkp * p.sw * 4, gt = (size_t)g.M * p.pxp * 4;
          at += wa > gt ? wa : gt;
        }
        p.off_goff = at;  // unused on the tensor path
      } else {
        p.off_goff = at;
        at += (size_t)g.M * p.ps * 4;
      }
      p.smem = at;
      if (best.smem == 0 || p.smem < best.smem) best = p;
      if (p.smem <= kSmemBudget) return p;
    }
  }
  return best;
}

__device__ __forceinline__ int pos_rc(int px, int TW) {
  const int r = px / TW;
  return (r << 16) | (px - r * TW);
}

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Raw bf16 bits of channel cl (relative to the slice) at staged offset pos.
__device__ __forceinline__ uint32_t staged_bits(const uint32_t* xs, int plane, int cl, int pos) {
  const uint32_t w = xs[(cl >> 1) * plane + pos];
  return (cl & 1) ? (w >> 16) : (w & 0xffffu);
}

// Offset-convolution backward of one band on tensor cores (bf16 operands,
// fp32 accumulation), two small GEMMs over the band's offset gradient goff:
//   weights: gw_off[m][(c,k)] += sum_px goff[m][px] * xbar[c](px + tap k)
//            (M = offset channels, N = (channel, tap), K = pixels)
//   input:   D[(c,k)][px] = sum_m w_off[m][c][k] * goff[m][px], added to the
//            grad_x window at the position tap k of pixel px reads
//            (M = (channel, tap), N = pixels, K = offset channels)
// Every mma.sync m16n8k16 fragment register is one 32-bit shared load: goff
// is kept as zero-padded bf16 pairs in both orientations (gA [m][px],
// gB [px][m]) and w_off^T as wA [(c,k)][m]; the staged input is read through
// a per-pixel position table (padding pixels point at a valid word and meet
// zero goff).
__device__ void offconv_bwd_mma(float* gw_off, const Geom& g, const Plan& pl,
                                const uint32_t* __restrict__ ga, const uint32_t* __restrict__ gb,
                                const uint32_t* __restrict__ wa, const uint32_t* __restrict__ xw,
                                float* gxs, const int* __restrict__ pos,
                                const int* __restrict__ tapoff, int c_begin, int ncur) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int M = g.M, PL = pl.plane;
  const int NK = ncur * g.K;
  constexpr int kWarps = kThreads / 32;
  const int mtiles = pl.mp16 / 16;

  // ---- weights: rows m, columns (c,k), reduction over pixels
  {
    const int ntiles = (NK + 7) / 8;
    const int ksteps = pl.pxp / 16;
    for (int nt = warp; nt < ntiles; nt += kWarps) {
      const int n = nt * 8 + gid;
      const int nc = n < NK ? n : NK - 1;
      const int cl = nc / g.K, k = nc - cl * g.K;
      const int toff = tapoff[k];
      const uint32_t* xc = xw + (cl >> 1) * PL;
      const int sh = (cl & 1) ? 16 : 0;
      float acc[5][4];
#pragma unroll
      for (int t = 0; t < 5; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
      for (int ks = 0; ks < ksteps; ++ks) {
        const int p0 = ks * 16 + 2 * tig;
        const uint32_t x0 = (xc[pos[p0] + toff] >> sh) & 0xffffu;
        const uint32_t x1 = (xc[pos[p0 + 1] + toff] >> sh) & 0xffffu;
        const uint32_t x2 = (xc[pos[p0 + 8] + toff] >> sh) & 0xffffu;
        const uint32_t x3 = (xc[pos[p0 + 9] + toff] >> sh) & 0xffffu;
        const uint32_t b0 = x0 | (x1 << 16), b1 = x2 | (x3 << 16);
#pragma unroll
        for (int mt = 0; mt < 5; ++mt) {
          if (mt >= mtiles) break;
          const uint32_t* a = ga + (mt * 16 + gid) * pl.sa + ks * 8 + tig;
          const uint32_t af[4] = {a[0], a[8 * pl.sa], a[4], a[8 * pl.sa + 4]};
          mma_bf16_16816(acc[mt], af, b0, b1);
        }
      }
#pragma unroll
      for (int mt = 0; mt < 5; ++mt) {
        if (mt >= mtiles) break;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int m = mt * 16 + gid + (h >> 1) * 8;
          const int nn = nt * 8 + 2 * tig + (h & 1);
          if (m < M && nn < NK) {
            const int ccl = nn / g.K, kk = nn - ccl * g.K;
            atomicAdd(gw_off + ((long long)m * g.c_in + c_begin + ccl) * g.K + kk, acc[mt][h]);
          }
        }
      }
    }
  }

  // ---- input: for each tap k, rows = channels, columns = pixels, reduction
  // over offset channels.  Within one tap the 32 lanes of an mma tile target
  // 32 distinct window positions (distinct channels or pixels), so the
  // shared-memory atomics of one instruction never collide.
  {
    const int ctiles = pl.cpc / 16;
    const int ptiles = pl.pxp / 8;
    const int ksteps = pl.mp16 / 16;
    for (int task = warp; task < g.K * ctiles; task += kWarps) {
      const int k = task / ctiles, ct = task - (task / ctiles) * ctiles;
      uint32_t af[5][4];
#pragma unroll
      for (int ks = 0; ks < 5; ++ks) {
        if (ks >= ksteps) break;
        const uint32_t* a = wa + (k * pl.cpc + ct * 16 + gid) * pl.sw + ks * 8 + tig;
        af[ks][0] = a[0];
        af[ks][1] = a[8 * pl.sw];
        af[ks][2] = a[4];
        af[ks][3] = a[8 * pl.sw + 4];
      }
      const int c0 = ct * 16 + gid, c1 = c0 + 8;  // accumulator rows (channels)
      const bool v0 = c0 < ncur, v1 = c1 < ncur;
      float* dst0 = gxs + c0 * PL + tapoff[k];
      float* dst1 = gxs + c1 * PL + tapoff[k];
      for (int nt = 0; nt < ptiles; ++nt) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t* b = gb + (nt * 8 + gid) * pl.sb + tig;
#pragma unroll
        for (int ks = 0; ks < 5; ++ks) {
          if (ks >= ksteps) break;
          mma_bf16_16816(acc, af[ks], b[ks * 8], b[ks * 8 + 4]);
        }
        const int px = nt * 8 + 2 * tig;
        if (px < pl.npx) {
          if (v0) atomicAdd(dst0 + pos[px], acc[0]);
          if (v1) atomicAdd(dst1 + pos[px], acc[2]);
        }
        if (px + 1 < pl.npx) {
          if (v0) atomicAdd(dst0 + pos[px + 1], acc[1]);
          if (v1) atomicAdd(dst1 + pos[px + 1], acc[3]);
        }
      }
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) k4_offconv_bwd(OffconvBwdArgs a, Plan pl) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr bool kBf16 = sizeof(T) == 2;
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
  int* pix = reinterpret_cast<int*>(smem + pl.off_tab);        // CUDA-core path: (row << 16 | col)
  const int tab_n = pl.pxp > PS ? pl.pxp : PS;
  int* tapoff = pix + tab_n;
  const bool tensor = kBf16 && M <= kOffconvMmaMaxM;

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

  if (tensor) {
    // positions of the band's pixels in the staged window (padding -> 0)
    int* pos = pix;
    for (int px = tid; px < pl.pxp; px += kThreads) {
      int v = 0;
      if (px < npx) {
        const int r = px / pl.TW;
        v = r * g.sh * pl.cols + (px - r * pl.TW) * g.sw;
      }
      pos[px] = v;
    }
    uint32_t* ga = reinterpret_cast<uint32_t*>(smem + pl.off_ga);
    uint32_t* gb = reinterpret_cast<uint32_t*>(smem + pl.off_gb);
    uint32_t* wa = reinterpret_cast<uint32_t*>(smem + pl.off_wa);
    // goff of the band (fp32) staged once, in wa's space before wa is built;
    // eight independent loads in flight per thread
    float* gtmp = reinterpret_cast<float*>(wa);  // [M][pxp]
    {
      constexpr int kB = 8;
      const int total = M * pl.pxp;
      for (int base = tid; base < total; base += kThreads * kB) {
        float v[kB];
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          const int idx = base + j * kThreads;
          v[j] = 0.f;
          if (idx < total) {
            const int m = idx / pl.pxp, px = idx - m * pl.pxp;
            if (px < npx) {
              const int e = pos_rc(px, pl.TW);
              const int ho = ho0 + (e >> 16), wo = wo0 + (e & 0xffff);
              if (ho < g.ho && wo < g.wo)
                v[j] = a.goff[((long long)n * M + m) * g.howo + (long long)ho * g.wo + wo];
            }
          }
        }
#pragma unroll
        for (int j = 0; j < kB; ++j)
          if (base + j * kThreads < total) gtmp[base + j * kThreads] = v[j];
      }
    }
    __syncthreads();
    auto pack = [](float lo, float hi) {
      __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
      return *reinterpret_cast<uint32_t*>(&v);
    };
    auto gv = [&](int m, int px) { return m < M ? gtmp[m * pl.pxp + px] : 0.f; };
    for (int idx = tid; idx < pl.mp16 * (pl.pxp / 2); idx += kThreads) {
      const int m = idx / (pl.pxp / 2), j = idx - m * (pl.pxp / 2);
      ga[m * pl.sa + j] = pack(gv(m, 2 * j), gv(m, 2 * j + 1));
    }
    for (int idx = tid; idx < pl.pxp * (pl.mp16 / 2); idx += kThreads) {
      const int px = idx / (pl.mp16 / 2), j = idx - px * (pl.mp16 / 2);
      gb[px * pl.sb + j] = pack(gv(2 * j, px), gv(2 * j + 1, px));
    }
    if (a.gb_off && slice == 0) {
      // one warp per offset channel: lane-strided sum, then a shuffle tree
      const int wp = tid >> 5, ln = tid & 31;
      for (int m = wp; m < M; m += kThreads / 32) {
        float s = 0.f;
        for (int px = ln; px < npx; px += 32) s += gtmp[m * pl.pxp + px];
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (ln == 0) atomicAdd(a.gb_off + m, s);
      }
    }
    __syncthreads();
    // w_off^T: rows (tap k, channel c), columns offset-channel pairs.  Each
    // offset channel's slice w_off[m][c_begin..][*] is contiguous in memory:
    // lanes run along it (coalesced), eight loads in flight per thread.
    {
      const __nv_bfloat16* wsrc = reinterpret_cast<const __nv_bfloat16*>(w_off);
      unsigned short* wh = reinterpret_cast<unsigned short*>(wa);  // bf16 halves
      for (int idx = tid; idx < pl.nkp * pl.sw; idx += kThreads) wa[idx] = 0u;
      __syncthreads();
      constexpr int kB = 8;
      const int span = ncur * g.K;  // contiguous elements per offset channel
      const int total = M * span;
      for (int base = tid; base < total; base += kThreads * kB) {
        unsigned short v[kB];
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          const int idx = base + j * kThreads;
          v[j] = 0;
          if (idx < total) {
            const int m = idx / span, t = idx - m * span;
            v[j] = (unsigned short)band::bf16_bits(wsrc + (long long)m * g.c_in * g.K +
                                                   (long long)c_begin * g.K + t);
          }
        }
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          const int idx = base + j * kThreads;
          if (idx < total) {
            const int m = idx / span, t = idx - m * span;
            const int cl = t / g.K, k = t - cl * g.K;
            wh[((k * pl.cpc + cl) * pl.sw) * 2 + m] = v[j];
          }
        }
      }
    }
    __syncthreads();
    offconv_bwd_mma(a.gw_off, g, pl, ga, gb, wa, xw, gxs, pos, tapoff, c_begin, ncur);
  } else {
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
    // tap, added to the window position that tap reads
    constexpr int kMc = 12;
    {
      const long long mstride = (long long)g.c_in * g.K;
      band::Walk2 w;
      w.init(tid, kThreads, npx);
      while (w.a < ncur) {
        const int cl = w.a, px = w.b;
        w.next();
        const int e = pix[px];
        const int pos = ((e >> 16) * g.sh + margin) * pl.cols + (e & 0xffff) * g.sw + margin;
        const T* wc = w_off + (long long)(c_begin + cl) * g.K;
        float* gp = gxs + cl * PL + pos;
        for (int m0 = 0; m0 < M; m0 += kMc) {
          float gv[kMc];
  #pragma unroll
          for (int t = 0; t < kMc; ++t) gv[t] = (m0 + t < M) ? goff[(m0 + t) * PS + px] : 0.f;
          for (int k = 0; k < g.K; ++k) {
            float s = 0.f;
  #pragma unroll
            for (int t = 0; t < kMc; ++t)
              if (m0 + t < M) s = __fmaf_rn(gv[t], ld_f(wc + (long long)(m0 + t) * mstride + k), s);
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

size_t offconv_bwd_smem_bytes(const Geom& g, dc_dtype dt) { return make_plan(g, dt).smem; }

cudaError_t launch_offconv_bwd(const OffconvBwdArgs& a, dc_dtype dt, cudaStream_t s) {
  const Plan pl = make_plan(a.g, dt);
  return dt == DC_BF16 ? launch_t<__nv_bfloat16>(a, pl, s) : launch_t<float>(a, pl, s);
}

}  // namespace dc
