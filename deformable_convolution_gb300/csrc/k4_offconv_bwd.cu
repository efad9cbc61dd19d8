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
constexpr size_t kSmemBudget = 72 * 1024;

struct Plan {
  int R, TW, tiles_w, tiles_h, npx;
  int ps;  // pixel stride of the per-band arrays
  int cpc, nslices;
  int rows, cols, plane;  // staged window: the band's receptive field
  size_t off_halo, off_gx, off_goff, off_tab, smem;
};

__host__ Plan make_plan(const Geom& g, dc_dtype dt) {
  const bool bf16 = dt == DC_BF16;
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
      size_t at = 0;
      p.off_halo = at;
      at += (size_t)(bf16 ? cpc / 2 : cpc) * p.plane * 4;
      p.off_gx = at;
      at += (size_t)cpc * p.plane * 4;
      p.off_goff = at;
      at += (size_t)g.M * p.ps * 4;
      p.off_tab = at;
      at += (size_t)(p.ps + g.K) * 4;
      p.smem = at;
      if (best.smem == 0 || p.smem < best.smem) best = p;
      if (p.smem <= kSmemBudget) return p;
    }
  }
  return best;
}

constexpr int kOffconvMmaMaxM = 80;

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
// mma.sync m16n8k16 fragments are built straight from shared memory (goff,
// the staged input) and from w_off in global memory (L1-resident slice).
// Needs M <= kOffconvMmaMaxM offset channels (five m16 tiles / k16 steps).
__device__ void offconv_bwd_mma(const __nv_bfloat16* __restrict__ w_off, float* gw_off,
                                const Geom& g, const Plan& pl, const float* goff,
                                const uint32_t* xw, float* gxs, const int* pix,
                                const int* tapoff, int c_begin, int ncur, int margin) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int M = g.M, PS = pl.ps, npx = pl.npx, PL = pl.plane;
  const int NK = ncur * g.K;  // (channel, tap) pairs of this slice
  const int window0 = margin * pl.cols + margin;
  constexpr int kWarps = kThreads / 32;

  // ---- weights: rows m, columns (c,k), reduction over pixels
  {
    const int mtiles = (M + 15) / 16;
    const int ntiles = (NK + 7) / 8;
    const int ksteps = (npx + 15) / 16;
    for (int nt = warp; nt < ntiles; nt += kWarps) {
      const int n = nt * 8 + gid;  // this lane's B column
      const int nc = n < NK ? n : NK - 1;
      const int cl = nc / g.K, k = nc - (nc / g.K) * g.K;
      const int toff = tapoff[k] + window0;
      float acc[5][4];
#pragma unroll
      for (int t = 0; t < 5; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
      for (int ks = 0; ks < ksteps; ++ks) {
        const int p0 = ks * 16 + 2 * tig;
        uint32_t xb[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int px = p0 + (h >> 1) * 8 + (h & 1);
          const int e = pix[px < npx ? px : npx - 1];
          const int pos = (e >> 16) * g.sh * pl.cols + (e & 0xffff) * g.sw + toff;
          xb[h] = px < npx ? staged_bits(xw, PL, cl, pos) : 0u;
        }
        const uint32_t b0 = xb[0] | (xb[1] << 16), b1 = xb[2] | (xb[3] << 16);
#pragma unroll
        for (int mt = 0; mt < 5; ++mt) {
          if (mt >= mtiles) break;
          const int m0 = mt * 16 + gid, m1 = m0 + 8;
          const int q0 = ks * 16 + 2 * tig, q1 = q0 + 8;
          auto gv = [&](int m, int q) { return (m < M && q < npx) ? goff[m * PS + q] : 0.f; };
          uint32_t af[4];
          af[0] = pack_bf16(gv(m0, q0), gv(m0, q0 + 1));
          af[1] = pack_bf16(gv(m1, q0), gv(m1, q0 + 1));
          af[2] = pack_bf16(gv(m0, q1), gv(m0, q1 + 1));
          af[3] = pack_bf16(gv(m1, q1), gv(m1, q1 + 1));
          mma_bf16_16816(acc[mt], af, b0, b1);
        }
      }
      // D rows m (gid, gid+8), columns (c,k) = nt*8 + 2*tig (+1)
#pragma unroll
      for (int mt = 0; mt < 5; ++mt) {
        if (mt >= mtiles) break;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int m = mt * 16 + gid + (h >> 1) * 8;
          const int nn = nt * 8 + 2 * tig + (h & 1);
          if (m < M && nn < NK) {
            const int ccl = nn / g.K, kk = nn - (nn / g.K) * g.K;
            atomicAdd(gw_off + ((long long)m * g.c_in + c_begin + ccl) * g.K + kk, acc[mt][h]);
          }
        }
      }
    }
  }

  // ---- input: rows (c,k), columns pixels, reduction over offset channels
  {
    const int mtiles = (NK + 15) / 16;
    const int ntiles = (npx + 7) / 8;
    const int ksteps = (M + 15) / 16;
    const long long mstride = (long long)g.c_in * g.K;
    for (int mt = warp; mt < mtiles; mt += kWarps) {
      const int r0 = mt * 16 + gid, r1 = r0 + 8;  // rows (c,k) of a0/a1
      const bool v0 = r0 < NK, v1 = r1 < NK;
      const int rc0 = v0 ? r0 : 0, rc1 = v1 ? r1 : 0;
      const __nv_bfloat16* w0 = w_off + (long long)(c_begin + rc0 / g.K) * g.K + rc0 % g.K;
      const __nv_bfloat16* w1 = w_off + (long long)(c_begin + rc1 / g.K) * g.K + rc1 % g.K;
      auto wv = [&](const __nv_bfloat16* base, bool valid, int m) -> uint32_t {
        return (valid && m < M) ? band::bf16_bits(base + (long long)m * mstride) : 0u;
      };
      uint32_t af[5][4];
#pragma unroll
      for (int ks = 0; ks < 5; ++ks) {
        if (ks >= ksteps) break;
        const int m = ks * 16 + 2 * tig;
        af[ks][0] = wv(w0, v0, m) | (wv(w0, v0, m + 1) << 16);
        af[ks][1] = wv(w1, v1, m) | (wv(w1, v1, m + 1) << 16);
        af[ks][2] = wv(w0, v0, m + 8) | (wv(w0, v0, m + 9) << 16);
        af[ks][3] = wv(w1, v1, m + 8) | (wv(w1, v1, m + 9) << 16);
      }
      // destination rows of this thread's accumulator values
      const int orow0 = mt * 16 + gid, orow1 = orow0 + 8;
      const int oc0 = orow0 < NK ? orow0 / g.K : 0, ok0 = orow0 < NK ? orow0 - oc0 * g.K : 0;
      const int oc1 = orow1 < NK ? orow1 / g.K : 0, ok1 = orow1 < NK ? orow1 - oc1 * g.K : 0;
      float* dst0 = gxs + oc0 * PL + tapoff[ok0] + window0;
      float* dst1 = gxs + oc1 * PL + tapoff[ok1] + window0;
      // four pixel tiles per round: all their loads and mma first, then the
      // round's shared-memory atomics
      constexpr int kNt = 4;
      for (int nt0 = 0; nt0 < ntiles; nt0 += kNt) {
        float acc[kNt][4];
#pragma unroll
        for (int tt = 0; tt < kNt; ++tt) {
          acc[tt][0] = acc[tt][1] = acc[tt][2] = acc[tt][3] = 0.f;
          const int q = (nt0 + tt) * 8 + gid;  // this lane's B column (pixel)
          const int qc = q < npx ? q : 0;
#pragma unroll
          for (int ks = 0; ks < 5; ++ks) {
            if (ks >= ksteps) break;
            const int m = ks * 16 + 2 * tig;
            auto gv = [&](int mm) { return (mm < M && q < npx) ? goff[mm * PS + qc] : 0.f; };
            const uint32_t b0 = pack_bf16(gv(m), gv(m + 1));
            const uint32_t b1 = pack_bf16(gv(m + 8), gv(m + 9));
            mma_bf16_16816(acc[tt], af[ks], b0, b1);
          }
        }
        // D: rows orow0/orow1, columns pixels nt*8 + 2*tig (+1)
#pragma unroll
        for (int tt = 0; tt < kNt; ++tt) {
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int px = (nt0 + tt) * 8 + 2 * tig + (h & 1);
            const bool row_ok = (h >> 1) ? orow1 < NK : orow0 < NK;
            if (!row_ok || px >= npx) continue;
            const int e = pix[px];
            const int pos = (e >> 16) * g.sh * pl.cols + (e & 0xffff) * g.sw;
            if (acc[tt][h] != 0.f) atomicAdd(((h >> 1) ? dst1 : dst0) + pos, acc[tt][h]);
          }
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
  float* goff = reinterpret_cast<float*>(smem + pl.off_goff);  // [M][PS]
  int* pix = reinterpret_cast<int*>(smem + pl.off_tab);
  int* tapoff = pix + PS;

  band::fill_pixel_table(pix, npx, pl.TW);
  for (int k = tid; k < g.K; k += kThreads) {
    const int i = k / g.kw;
    tapoff[k] = i * g.dh * pl.cols + (k - i * g.kw) * g.dw;
  }
  band::stage_window<T>(x, g, img, c_begin, pl.cpc, ylo, xlo, pl.rows, pl.cols, PL, xw);
  for (int idx = tid; idx < pl.cpc * PL; idx += kThreads) gxs[idx] = 0.f;
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

  if (kBf16 && M <= kOffconvMmaMaxM) {
    offconv_bwd_mma(reinterpret_cast<const __nv_bfloat16*>(w_off), a.gw_off, g, pl, goff, xw,
                    gxs, pix, tapoff, c_begin, ncur, margin);
  } else {
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
    }
  if (a.gb_off && slice == 0) {
    for (int m = tid; m < M; m += kThreads) {
      float s = 0.f;
      for (int px = 0; px < npx; ++px) s += goff[m * PS + px];
      atomicAdd(a.gb_off + m, s);
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
  dim3 grid((unsigned)(pl.nslices * pl.tiles_w), (unsigned)pl.tiles_h, (unsigned)a.g.n);
  kern<<<grid, kThreads, pl.smem, s>>>(a, pl);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace

size_t offconv_bwd_smem_bytes(const Geom& g, dc_dtype dt) { return make_plan(g, dt).smem; }

cudaError_t launch_offconv_bwd(const OffconvBwdArgs& a, dc_dtype dt, cudaStream_t s) {
  const Plan pl = make_plan(a.g, dt);
  return dt == DC_BF16 ? launch_t<__nv_bfloat16>(a, pl, s) : launch_t<float>(a, pl, s);
}

}  // namespace dc
