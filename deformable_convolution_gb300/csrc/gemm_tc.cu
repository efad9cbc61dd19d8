// Main-convolution GEMMs on the 5th-generation tensor cores (bf16 inputs,
// fp32 accumulation in tensor memory).
//
// Explainer page "DefT: Boosting Scalability of Deformable Convolution
// Operations on GPUs", "The argument in one glance / This paper's idea" and
// "The idea": the main convolution over the deformed map is left as a dense
// GEMM -- the one step of the layer that is a true contraction.  On GB300 it
// runs here as a hand-written tcgen05 kernel instead of a library call.
// With the column layout col[kdim][image][pixel]:
//   FWD   y[b][o][q]    = sum_r   w[o][r]  * col[r][b][q]     A = w   (K-major)
//                                                              B = col (MN-major)
//   GCOL  gcol[r][b][q] = sum_o   w[o][r]  * gy[b][o][q]      A = w^T (MN-major)
//                                                              B = gy  (MN-major)
//   GW    gw[o][r]     += sum_b,q gy[b][o][q] * col[r][b][q]  A = gy  (K-major)
//                                                              B = col (K-major)
// One CTA computes one 128 x BN output tile (GW: one K-split of it).
// Warp roles: warps 0-3 read the accumulator out of tensor memory (one TMEM
// lane quarter each), warp 4 issues TMA loads into a ring of shared-memory
// stages, warp 5 issues tcgen05.mma (one thread) and commits each stage back to
// the producer.  All operand tiles use the 128-byte swizzle.  Every mbarrier
// wait is bounded: on expiry the kernel raises the library's device error flag,
// skips the rest of its work, frees its tensor memory and returns.
#include <cuda.h>

#include <cooperative_groups.h>

#include "dc_common.cuh"

namespace dc {

__device__ unsigned int g_dc_device_error;

namespace {

constexpr int kBM = 128, kBK = 64;
constexpr int kThreads = 192;
constexpr uint32_t kSpinLimit = 1u << 24;
// FWD / GCOL / GW work on the plane-major deformed map col[c*K + tap][n][pixel];
// FWDC / GCOLC / GWC on the pixel-major one, col[n][pixel][tap][channel], with
// the main weights permuted to w'[o][tap][channel] (the channels-last path):
//   FWDC   y[b][o][q]       = sum_r w'[o][r] * col[b][q][r]     A = w'  (K-major)
//                                                               B = col (K-major)
//   GCOLC  gcol[b][q][r]    = sum_o gy[b][o][q] * w'[o][r]      A = gy  (MN-major, M = pixels)
//                                                               B = w'  (MN-major)
//   GWC    gw[o][c][tap]   += sum_b,q gy[b][o][q] * col[b][q][r], r = tap*C + c
//                                                               A = gy  (K-major)
//                                                               B = col (MN-major)
enum Kind { FWD = 0, GCOL = 1, GW = 2, FWDC = 3, GCOLC = 4, GWC = 5 };
constexpr bool is_fwd(int k) { return k == FWD || k == FWDC; }
constexpr bool is_gcol(int k) { return k == GCOL || k == GCOLC; }
constexpr bool is_gw(int k) { return k == GW || k == GWC; }

struct TcArgs {
  int c_out, kdim, howo, nimg;
  int kb_total;          // k-blocks of the whole reduction
  int kb_per_split;      // GW: k-blocks per CTA along blockIdx.z
  int qblocks;           // GW: k-blocks per image (ceil(howo / 64))
  int fwd_split;         // FWD: 2 = the k-blocks are split over a 2-CTA cluster along y
  void* out;
  long long out_row, out_img;  // GCOL: gcol pitches (elements)
  ZeroArgs zero;               // GCOL: the backward's atomic targets, cleared by warps 0-3
  float* gmax;                 // GCOL: max |gcol| of each tile, one float per epilogue warp
  const float* gwo_img;        // GW: per-image grad_w_off partials to sum after K4 (or null)
  float* gw_off;
  long long gwo_count;         // floats per image
  int gwo_nimg, gwo_m, gwo_cin, gwo_k;  // images; M, C_in, K of the partials' order
  int cin, ktaps;              // GWC: C_in and taps, to map columns (tap, c) to grad_w[o][c][tap];
                               // cin = 0: add in w' order ([o][tap][c], float4 atomics)
  // the tile grid (x: column tiles, y: row tiles, z: images or splits); a
  // persistent launch runs tiles blockIdx.x, + gridDim.x, ... of it
  int vgx, vgy, vgz, persistent;
  int flat;  // FWDC: column tiles run over the flat pixel index b * howo + q of all images
  int relu;  // FWD / FWDC: y = max(y, 0) in the epilogue
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait; false (and the device error flag raised) on expiry.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  atomicOr(&g_dc_device_error, 1u);
  return false;
}

__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                       int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                       int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// ReLU on 32 fp32 values in place (the forward's fused activation): positive
// values and NaN kept, everything else (-0 included) +0.
__device__ __forceinline__ void relu32(uint32_t* r) {
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float v = __uint_as_float(r[j]);
    if (!(v > 0.f) && v == v) r[j] = 0u;
  }
}

// Row m of y (bf16), columns n_first .. n_first + 31, from 32 fp32 values.
__device__ __forceinline__ void store_y_row(__nv_bfloat16* dst, const uint32_t* r, int n_first,
                                            int howo) {
  if (n_first + 32 <= howo) {
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      uint4 pk;
      uint32_t* pw = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(r[v * 8 + 2 * e]),
                                                  __uint_as_float(r[v * 8 + 2 * e + 1]));
        pw[e] = *reinterpret_cast<uint32_t*>(&b2);
      }
      *reinterpret_cast<uint4*>(dst + v * 8) = pk;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (n_first + j < howo) dst[j] = __float2bfloat16_rn(__uint_as_float(r[j]));
  }
}

// TMA store of a shared-memory box (bulk-group completion).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1,
                                             int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(map),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_store_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void tma_store_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: 128-byte swizzle, sm_100 descriptor version.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, M = 128, N = bn.
__host__ __device__ constexpr uint32_t idesc_bf16(int bn, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                     uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// MH = 2: one CTA computes 256 rows of the output (two M = 128 halves, two
// accumulators side by side in tensor memory) against one B tile, so the
// large B operand (the deformed map) is read once instead of once per half.
template <int KIND, int BN, int MH = 1, int NACC = 2>
struct Cfg {
  static constexpr int kAHalf = kBM * kBK * 2;
  static constexpr int kABytes = MH * kAHalf;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStage = kABytes + kBBytes;
  // GCOL reduces over C_out only (a few k-blocks): two stages, so that three
  // CTAs fit on an SM; the long reductions keep a deeper ring.
  // GCOL has two k-blocks; four stages let two FWD CTAs share an SM
  // (as many as fit, up to four, for the wide single-wave tiles)
  static constexpr int kStages =
      is_gcol(KIND) ? (BN == 256 ? 3 : 2) : ((225 * 1024) / kStage < 4 ? (225 * 1024) / kStage : 4);
  // tensor-memory columns of one half's accumulator: BN rounded up to a
  // power of two; NACC accumulators (two: the epilogue of one tile overlaps
  // the next tile's MMAs; one: wide tiles of a single-wave launch), allocated
  // as a power of two
  static constexpr int kHS = BN <= 32 ? 32 : (BN <= 64 ? 64 : (BN <= 128 ? 128 : 256));
  static constexpr int kTmemCols = NACC * MH * kHS;
  static_assert(kTmemCols <= 512, "tensor memory holds 512 columns");
  // GCOL's bf16 store staging: 4 warps x BN/64 boxes of 32 x 64
  static constexpr int kStg = is_gcol(KIND) ? 4 * (BN / 64) * 4096 : 0;
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStage + kStg + 256;
  static constexpr int kAMn = is_gcol(KIND) ? 1 : 0;
  static constexpr int kBMn = (KIND == GW || KIND == FWDC) ? 0 : 1;
};

template <int KIND, int BN, int MH = 1, int NACC = 2>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            const __grid_constant__ CUtensorMap tmC, TcArgs a) {
  using C = Cfg<KIND, BN, MH, NACC>;
  static_assert(MH == 1 || KIND == FWDC || KIND == GWC, "two M halves: forward and weight-gradient kinds");
  constexpr uint32_t kAcc = MH * C::kHS;  // tensor-memory columns of one accumulator
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* stg = smem + C::kStages * C::kStage;  // GCOL store staging
  uint64_t* full = reinterpret_cast<uint64_t*>(stg + C::kStg);
  uint64_t* empty = full + C::kStages;
  uint64_t* tfull = empty + C::kStages;  // accumulator b complete (MMA -> epilogue)
  uint64_t* tempty = tfull + 2;          // accumulator b drained (epilogue -> MMA)
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tempty + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // FWD split over a 2-CTA cluster: rank 0 takes the first half of the
  // k-blocks, rank 1 the second; rank 1 hands its fp32 tile to rank 0 through
  // distributed shared memory and rank 0 writes y (one tile per CTA)
  const bool split = is_fwd(KIND) && a.fwd_split == 2;
  const int rank = split ? (int)(blockIdx.y & 1) : 0;
  const int ntiles =
      a.persistent ? (a.vgx * a.vgy * a.vgz - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 1;
  struct Tile {
    int bx, by, m0, n0, z, kb_begin, nkb;
  };
  // this CTA's j-th tile
  auto tile = [&](int j) {
    Tile T;
    if (a.persistent) {
      const int t = (int)blockIdx.x + j * (int)gridDim.x;
      T.bx = t % a.vgx;
      const int r = t / a.vgx;
      T.by = r % a.vgy;
      T.z = r / a.vgy;
    } else {
      T.bx = blockIdx.x;
      T.by = blockIdx.y;
      T.z = blockIdx.z;
    }
    T.m0 = (split ? (T.by >> 1) : T.by) * kBM * MH;
    T.n0 = T.bx * BN;
    int kb_begin = 0, kb_end = a.kb_total;
    if (is_gw(KIND)) {
      kb_begin = T.z * a.kb_per_split;
      kb_end = min(a.kb_total, kb_begin + a.kb_per_split);
    }
    if (split) {
      const int half = (a.kb_total + 1) / 2;
      kb_begin = rank ? half : 0;
      kb_end = rank ? a.kb_total : half;
    }
    T.kb_begin = kb_begin;
    T.nkb = kb_end > kb_begin ? kb_end - kb_begin : 0;
    return T;
  };
  bool ok = true;  // no wait expired

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"((uint32_t)C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);  // one arrival per epilogue warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // The forward GEMM reads the column K1 writes; GCOL, the first kernel of
  // the backward call, waits for whatever precedes it on the stream.
  // The weight-gradient GEMM follows K4 but reads nothing K4 writes: it starts
  // only once every K4 block has passed its own wait on K3 (which replays the
  // column it reads, after GCOL cleared grad_w), so it runs beside K4 and
  // waits for K4 only before it exits.
  if (!is_gw(KIND)) pdl_wait();

  if (warp == 4) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      int it = 0;  // k-blocks issued so far (all tiles): ring slot and phase
      for (int j = 0; j < ntiles && ok; ++j) {
        const Tile T = tile(j);
        const int m0 = T.m0, n0 = T.n0, z = T.z;
        for (int i = 0; i < T.nkb; ++i, ++it) {
          const int s = it % C::kStages;
          if (it >= C::kStages && !mbar_wait(&empty[s], ((it / C::kStages) - 1) & 1)) {
            ok = false;
            break;
          }
          unsigned char* sa = smem + s * C::kStage;
          unsigned char* sb = sa + C::kABytes;
          mbar_expect_tx(&full[s], C::kStage);
          const int kb = T.kb_begin + i;
          if (KIND == FWD) {
            tma_2d(sa, &tmA, &full[s], kb * kBK, m0);
#pragma unroll
            for (int h = 0; h < BN / 64; ++h) tma_3d(sb + h * 8192, &tmB, &full[s], n0 + 64 * h, z, kb * kBK);
          } else if (KIND == FWDC) {
            // A: w' rows m0.. (and m0 + 128..), k-block kb; B: BN pixels of image z, k-block kb
            tma_2d(sa, &tmA, &full[s], kb * kBK, m0);
            if (MH == 2) tma_2d(sa + C::kAHalf, &tmA, &full[s], kb * kBK, m0 + kBM);
            if (a.flat)
              tma_2d(sb, &tmB, &full[s], kb * kBK, n0);
            else
              tma_3d(sb, &tmB, &full[s], kb * kBK, n0, z);
          } else if (KIND == GCOLC) {
            // A: grad_y rows kb*64.. (output channels) x 128 pixels of image z,
            // as two 64-pixel MN chunks; B: w' rows kb*64.. x BN columns
            tma_3d(sa, &tmA, &full[s], m0, kb * kBK, z);
            tma_3d(sa + 8192, &tmA, &full[s], m0 + 64, kb * kBK, z);
#pragma unroll
            for (int h = 0; h < BN / 64; ++h) tma_2d(sb + h * 8192, &tmB, &full[s], n0 + 64 * h, kb * kBK);
          } else if (KIND == GWC) {
            const int img = kb / a.qblocks, q0 = (kb - img * a.qblocks) * kBK;
            tma_3d(sa, &tmA, &full[s], q0, m0, img);
            if (MH == 2) tma_3d(sa + C::kAHalf, &tmA, &full[s], q0, m0 + kBM, img);
#pragma unroll
            for (int h = 0; h < BN / 64; ++h) tma_3d(sb + h * 8192, &tmB, &full[s], n0 + 64 * h, q0, img);
          } else if (KIND == GCOL) {
            tma_2d(sa, &tmA, &full[s], m0, kb * kBK);
            tma_2d(sa + 8192, &tmA, &full[s], m0 + 64, kb * kBK);
#pragma unroll
            for (int h = 0; h < BN / 64; ++h) tma_3d(sb + h * 8192, &tmB, &full[s], n0 + 64 * h, kb * kBK, z);
          } else {
            const int img = kb / a.qblocks, q0 = (kb - img * a.qblocks) * kBK;
            tma_3d(sa, &tmA, &full[s], q0, m0, img);
            tma_3d(sb, &tmB, &full[s], q0, img, n0);
          }
        }
      }
    }
    pdl_release();
  } else if (warp == 5) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = idesc_bf16(BN, C::kAMn, C::kBMn);
      int it = 0;
      for (int j = 0; j < ntiles && ok; ++j) {
        const Tile T = tile(j);
        const int b = j % NACC;
        // accumulator b was drained by the epilogue (its use NACC tiles ago)
        if (j >= NACC && !mbar_wait(&tempty[b], ((j / NACC) - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)b * kAcc;
        for (int i = 0; i < T.nkb; ++i, ++it) {
          const int s = it % C::kStages;
          if (!mbar_wait(&full[s], (it / C::kStages) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * C::kStage);
          const uint32_t sb = sa + C::kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // K-major: step 32 bytes inside the 128-byte swizzled row;
            // MN-major: step 16 k-rows = two 1024-byte swizzle atoms
            const uint64_t db = C::kBMn ? sdesc(sb + kk * 2048, 8192, 1024) : sdesc(sb + kk * 32, 16, 1024);
#pragma unroll
            for (int h = 0; h < MH; ++h) {
              const uint32_t sah = sa + h * C::kAHalf;
              const uint64_t da = C::kAMn ? sdesc(sah + kk * 2048, 8192, 1024) : sdesc(sah + kk * 32, 16, 1024);
              umma(acc + h * C::kHS, da, db, idesc, (i > 0 || kk > 0) ? 1u : 0u);
            }
          }
          umma_commit(&empty[s]);
        }
        umma_commit(&tfull[b]);  // arrives once the tile's MMAs are complete
      }
    }
    pdl_release();
  } else {
    // -------------------------------------------------------------- epilogue (warps 0-3)
    if (is_gcol(KIND)) {
      // before the first accumulator is ready, clear this CTA's share of the
      // buffers the rest of the backward pass accumulates into with atomics
      const long long nparts = (long long)gridDim.x * gridDim.y * gridDim.z;
      const long long part = blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y * blockIdx.z);
      zero_share(a.zero, part, nparts, threadIdx.x, 128);
    }
    const int row = warp * 32 + lane;
    for (int j = 0; j < ntiles; ++j) {
      const Tile T = tile(j);
      const int m0 = T.m0, n0 = T.n0, z = T.z, nkb = T.nkb;
      const int b = j % NACC;
      ok = ok && __all_sync(0xffffffffu, mbar_wait(&tfull[b], (j / NACC) & 1));
      if (!ok) break;
      tc_fence_after();
      if (is_gcol(KIND)) {
        // the staging buffers' previous TMA stores have read them
        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        __syncwarp();
      }
      // GCOL: bits of the largest |value| this thread stores; as integers the
      // magnitudes order like the floats, and inf / NaN sort above every finite value
      uint32_t amax = 0u;
      // One tile in this CTA (the weight-gradient GEMM's splits): once its
      // accumulator is complete the operand ring is idle, and the tile's
      // float4 atomics (w' order) go through it: each warp stages 32 rows x
      // 128 bytes (row l at l * 128, 16-byte piece v at (v ^ (l & 7)) * 16: no
      // bank conflicts) and reads them back eight lanes per row, so every
      // vector atomic instruction covers four whole 128-byte lines instead of
      // 32 rows.  (The forward GEMM's bf16 stores measured slower this way.)
      const bool staged = KIND == GWC && ntiles == 1 && nkb > 0 && a.cin == 0;
      if (staged) {
        unsigned char* wst = smem + warp * 4096;
        const uint32_t tb0 = tmem + (uint32_t)b * kAcc + ((uint32_t)(warp * 32) << 16);
        float* gwo = static_cast<float*>(a.out);
#pragma unroll 1
        for (int hc = 0; hc < MH * (BN / 32); ++hc) {
          const int h = hc / (BN / 32), c = hc - h * (BN / 32);
          uint32_t r[32];
          tmem_ld32(tb0 + (uint32_t)(h * C::kHS) + (uint32_t)(c * 32), r);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            *reinterpret_cast<uint4*>(wst + lane * 128 + ((v ^ (lane & 7)) << 4)) =
                make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
          __syncwarp();
          const int pc = lane & 7;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = (lane >> 3) + 4 * i;
            const float4 val = *reinterpret_cast<const float4*>(wst + rr * 128 + ((pc ^ (rr & 7)) << 4));
            const int mm = m0 + h * kBM + warp * 32 + rr;
            const int col = n0 + c * 32 + pc * 4;  // kdim is a multiple of 4
            if (mm < a.c_out && col < a.kdim)
              atomicAdd(reinterpret_cast<float4*>(gwo + (long long)mm * a.kdim + col), val);
          }
          __syncwarp();
        }
      }
#pragma unroll 1
      for (int hc = 0; !staged && hc < MH * (BN / 32); ++hc) {
        // half h (rows m0 + 128 h ..) of the output, its column chunk c
        const int h = hc / (BN / 32), c = hc - h * (BN / 32);
        const int m = m0 + h * kBM + row;
        const uint32_t tbase = tmem + (uint32_t)b * kAcc + (uint32_t)(h * C::kHS) + ((uint32_t)(warp * 32) << 16);
        uint32_t r[32];
        tmem_ld32(tbase + c * 32, r);
        if (nkb == 0) continue;
        const int n_first = n0 + c * 32;
        if (is_fwd(KIND) && split) {
          // rank 1: its partial tile to its own shared memory, column-major
          // (lanes write consecutive words); rank 0 combines after the cluster
          // barrier below
          if (rank == 1) {
            float* part = reinterpret_cast<float*>(smem);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) part[(c * 32 + jj) * kBM + row] = __uint_as_float(r[jj]);
          }
        } else if (is_fwd(KIND) && a.flat) {
          // flat pixel index f = b * howo + q over all images
          if (m >= a.c_out) continue;
          if (a.relu) relu32(r);
          const long long total = (long long)a.nimg * a.howo;
          if (n_first >= total) continue;
          const int zb = n_first / a.howo, q = n_first - zb * a.howo;
          __nv_bfloat16* y = static_cast<__nv_bfloat16*>(a.out);
          if (q + 32 <= a.howo) {
            store_y_row(y + ((long long)zb * a.c_out + m) * a.howo + q, r, q, a.howo);
          } else {
            // the chunk crosses into the next image (or past the last pixel)
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              const int qj = q + jj;
              const bool next = qj >= a.howo;
              if (n_first + jj < total)
                y[((long long)(zb + (next ? 1 : 0)) * a.c_out + m) * a.howo + (next ? qj - a.howo : qj)] =
                    __float2bfloat16_rn(__uint_as_float(r[jj]));
            }
          }
        } else if (is_fwd(KIND)) {
          if (m >= a.c_out) continue;
          if (a.relu) relu32(r);
          store_y_row(static_cast<__nv_bfloat16*>(a.out) + ((long long)z * a.c_out + m) * a.howo + n_first,
                      r, n_first, a.howo);
        } else if (is_gcol(KIND)) {
          // gcol leaves as bf16: this warp's 32 rows x 64 columns go through
          // its staging buffer in the 128-byte swizzled layout of the store
          // map, one TMA store per two 32-column chunks; rows and columns
          // beyond the tensor are clipped by the TMA unit.  The magnitude
          // bound is taken before rounding.
          if (KIND == GCOL && m < a.kdim) {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
              if (n_first + jj < a.howo) amax = max(amax, r[jj] & 0x7fffffffu);
          }
          unsigned char* buf = stg + (warp * (BN / 64) + (c >> 1)) * 4096;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 pk;
            uint32_t* pw = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(r[v * 8 + 2 * e]),
                                                        __uint_as_float(r[v * 8 + 2 * e + 1]));
              pw[e] = *reinterpret_cast<uint32_t*>(&b2);
            }
            const int piece = (c & 1) * 4 + v;  // 16-byte piece of the 128-byte row
            *reinterpret_cast<uint4*>(buf + lane * 128 + ((piece ^ (lane & 7)) << 4)) = pk;
          }
          if (c & 1) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            const int box_n = n0 + (c >> 1) * 64;
            if (KIND == GCOL && lane == 0 && m0 + warp * 32 < a.kdim && box_n < a.howo) {
              tma_store_3d(&tmC, buf, box_n, z, m0 + warp * 32);
              tma_store_commit();
            }
            // pixel-major: rows are pixels, columns (tap, channel)
            if (KIND == GCOLC && lane == 0 && m0 + warp * 32 < a.howo && box_n < a.kdim) {
              tma_store_3d(&tmC, buf, box_n, m0 + warp * 32, z);
              tma_store_commit();
            }
          }
        } else if (KIND == GWC && a.cin > 0) {
          if (m >= a.c_out) continue;
          // column r = tap * C + c of w' is grad_w[m][c][tap]
          float* dst = static_cast<float*>(a.out) + (long long)m * a.kdim;
          int tap = n_first / a.cin, cc = n_first - tap * a.cin;
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            if (n_first + jj < a.kdim) atomicAdd(dst + (long long)cc * a.ktaps + tap, __uint_as_float(r[jj]));
            if (++cc == a.cin) {
              cc = 0;
              ++tap;
            }
          }
        } else {
          if (m >= a.c_out) continue;
          float* dst = static_cast<float*>(a.out) + (long long)m * a.kdim + n_first;
          if (n_first + 32 <= a.kdim) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              atomicAdd(reinterpret_cast<float4*>(dst + v * 4),
                        make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                    __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3])));
          } else {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
              if (n_first + jj < a.kdim) atomicAdd(dst + jj, __uint_as_float(r[jj]));
          }
        }
      }
      // accumulator b is free for the tile after next (the split forward
      // reads its only tile once more below; it has no next tile)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[b]);
      if (KIND == GCOL && a.gmax) {
        for (int o = 16; o > 0; o >>= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const long long t = T.bx + (long long)a.vgx * (T.by + (long long)a.vgy * z);
        if (lane == 0) a.gmax[t * 4 + warp] = __uint_as_float(amax);
      }
    }
    if (is_gcol(KIND) && lane == 0) tma_store_wait_all();  // gcol written before exit
    pdl_release();
  }
  if (is_fwd(KIND) && split) {
    // every thread of both CTAs: rank 1's partial is in its shared memory
    cooperative_groups::cluster_group cluster = cooperative_groups::this_cluster();
    cluster.sync();
    if (rank == 0 && warp < 4) {
      const Tile T = tile(0);
      const int m0 = T.m0, n0 = T.n0, z = T.z, nkb = T.nkb;
      const float* peer = cluster.map_shared_rank(reinterpret_cast<float*>(smem), 1);
      const int row = warp * 32 + lane;
      const int m = m0 + row;
      const uint32_t tbase = tmem + ((uint32_t)(warp * 32) << 16);
      const bool peer_ok = nkb > 0 && a.kb_total > (a.kb_total + 1) / 2;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tbase + c * 32, r);
        if (!ok) continue;
        if (peer_ok) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            r[j] = __float_as_uint(__uint_as_float(r[j]) + peer[(c * 32 + j) * kBM + row]);
        }
        const int n_first = n0 + c * 32;
        if (a.relu) relu32(r);
        if (m < a.c_out)
          store_y_row(static_cast<__nv_bfloat16*>(a.out) + ((long long)z * a.c_out + m) * a.howo + n_first,
                      r, n_first, a.howo);
      }
    }
    cluster.sync();  // rank 0 is done reading rank 1's shared memory
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"((uint32_t)C::kTmemCols)
                 : "memory");
  if (is_gw(KIND)) {
    pdl_wait();  // completes no earlier than K4
    if (a.gwo_img) {
      // K4 is complete: sum its per-image grad_w_off partials, float4 runs of
      // K4's accumulator order spread over all CTAs of this grid, each element
      // stored to its place in grad_w_off (the buffer is 16-byte aligned and
      // the count a multiple of 4: checked on the host)
      const long long c4 = a.gwo_count / 4;
      const long long nthreads = (long long)gridDim.x * gridDim.y * gridDim.z * kThreads;
      const long long me =
          ((long long)blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y * blockIdx.z)) *
              kThreads + threadIdx.x;
      const float4* src = reinterpret_cast<const float4*>(a.gwo_img);
      for (long long e = me; e < c4; e += nthreads) {
        // eight images' loads in flight per thread
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        for (int n0 = 0; n0 < a.gwo_nimg; n0 += 8) {
          float4 v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            v[u] = n0 + u < a.gwo_nimg ? src[(long long)(n0 + u) * c4 + e] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            s[0] += v[u].x;
            s[1] += v[u].y;
            s[2] += v[u].z;
            s[3] += v[u].w;
          }
        }
        long long d[4];
        gwo_frag_dest4((int)e, a.gwo_m, a.gwo_cin, a.gwo_k, d);
#pragma unroll
        for (int h = 0; h < 4; ++h)
          if (d[h] >= 0) a.gw_off[d[h]] = s[h];
      }
    }
  }
}

// ---------------------------------------------------------------- sampled forward GEMM
// The forward main convolution with its B operand -- the deformed map --
// produced in shared memory by sampling warps instead of read from a column
// buffer in HBM: the three operators of "The argument in one glance" in fewer
// kernels, the fusion the explainer page argues against because the GEMM
// stops being a library call ("Why it fell short", "This paper's idea"), built
// here as a measured alternative.  One CTA computes a 128 x 64 tile of y.  Per
// 64-row k-block, warp 4 loads the weight tile with TMA, the ten sampling
// warps (0-3 and 6-11) write the 64 x 64 bf16 map tile in the 128-byte
// swizzled MN-major layout a TMA load of the column would have produced, and
// warp 5 issues the MMAs; warps 0-3 then drain the accumulator.  The samples
// use the offsets the offset convolution wrote (staged once per CTA) and read
// x's four corners from global memory with the fused stage's arithmetic, so
// the map values and the MMA sequence are those of the two-kernel path.
constexpr int kFsThreads = 384;
constexpr int kFsSampleWarps = 10;
constexpr int kFsStages = 4;
constexpr int kFsBN = 64;

struct FsArgs {
  Geom g;
  const __nv_bfloat16* x;
  const float* off;  // [n][M][howo]
  __nv_bfloat16* y;  // [n][c_out][howo]
  int kb_total;
};

__host__ __device__ inline size_t fs_smem_bytes(int M) {
  return 1024 + (size_t)kFsStages * Cfg<FWD, kFsBN>::kStage + (size_t)M * kFsBN * 4 +
         (size_t)kFsBN * 8 + 256;
}

__device__ __forceinline__ float corner(const __nv_bfloat16* plane, const Geom& g, int y, int x) {
  return (y >= 0 && y < g.h && x >= 0 && x < g.w) ? __bfloat162float(plane[(long long)y * g.w + x])
                                                  : 0.0f;
}

__global__ void __launch_bounds__(kFsThreads, 1)
    tc_fwd_sampled(const __grid_constant__ CUtensorMap tmA, FsArgs a) {
  using C = Cfg<FWD, kFsBN>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Geom g = a.g;
  float* offs = reinterpret_cast<float*>(smem + kFsStages * C::kStage);  // [M][64]
  int2* base = reinterpret_cast<int2*>(offs + (size_t)g.M * kFsBN);      // tap-0 row, column per pixel
  uint64_t* full = reinterpret_cast<uint64_t*>(base + kFsBN);
  uint64_t* empty = full + kFsStages;
  uint64_t* done = empty + kFsStages;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kFsBN, n = blockIdx.z;
  const int nkb = a.kb_total;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"((uint32_t)C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < kFsStages; ++s) {
      mbar_init(&full[s], 1 + kFsSampleWarps);  // the TMA's expect_tx + one per sampling warp
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  pdl_wait();  // the offsets come from the offset convolution just before
  for (int idx = threadIdx.x; idx < g.M * kFsBN; idx += kFsThreads) {
    const int m = idx / kFsBN, p = idx - m * kFsBN;
    offs[idx] = n0 + p < g.howo ? a.off[((long long)n * g.M + m) * g.howo + n0 + p] : 0.f;
  }
  for (int p = threadIdx.x; p < kFsBN; p += kFsThreads) {
    const int q = n0 + p, ho = q / g.wo, wo = q - ho * g.wo;
    base[p] = make_int2(ho * g.sh - g.ph, wo * g.sw - g.pw);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_release();
  const uint32_t tmem = *tmem_holder;
  bool ok = true;

  if (warp == 4) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer (weights)
      for (int i = 0; i < nkb; ++i) {
        const int s = i % kFsStages;
        if (i >= kFsStages && !mbar_wait(&empty[s], ((i / kFsStages) - 1) & 1)) break;
        mbar_expect_tx(&full[s], C::kABytes);
        tma_2d(smem + s * C::kStage, &tmA, &full[s], i * kBK, m0);
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = idesc_bf16(kFsBN, 0, 1);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % kFsStages;
        if (!mbar_wait(&full[s], (i / kFsStages) & 1)) break;
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + s * C::kStage);
        const uint32_t sb = sa + C::kABytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          umma(tmem, sdesc(sa + kk * 32, 16, 1024), sdesc(sb + kk * 2048, 8192, 1024), idesc,
               (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&empty[s]);
      }
      umma_commit(done);
    }
  } else {
    // -------------------------------------------------------------- sampling warps
    // The block's 64 k rows are (channel, tap) pairs in the weights' order
    // k = c * K + tap.  A warp takes a (tap, 32-pixel half) item: lane l owns
    // pixel l (+ 32), computes that tap's sampling point once per offset
    // group and blends it for every channel of the block that has a row for
    // the tap, storing each value at its place in the row's swizzled 16-byte
    // chunks.  The corner loads of one instruction fall on neighbouring pixels.
    constexpr int kH = kFsBN / 32;
    const int sw = warp < 4 ? warp : warp - 2;
    const __nv_bfloat16* ximg = a.x + (long long)n * g.c_in * g.hw;
    for (int i = 0; i < nkb; ++i) {
      const int s = i % kFsStages;
      if (i >= kFsStages) {
        const bool w_ok = mbar_wait(&empty[s], ((i / kFsStages) - 1) & 1);
        if (!__all_sync(0xffffffffu, w_ok)) {
          ok = false;
          break;
        }
      }
      unsigned char* sb = smem + s * C::kStage + C::kABytes;
      const int k_first = i * kBK;
      const int k_last = min(g.kdim, k_first + kBK) - 1;
      for (int item = sw; item < g.K * kH; item += kFsSampleWarps) {
        const int tap = item / kH, h = item - tap * kH;
        const int p = lane + 32 * h;
        const int ti = tap / g.kw, tj = tap - ti * g.kw;
        const bool px_ok = n0 + p < g.howo;
        const int2 b = base[p];
        // channels whose row c * K + tap lies in [k_first, k_last], in runs
        // of one offset group (one sampling point) and chunks of eight whose
        // corner loads are all issued before the first blend
        const int c_lo = (k_first - tap + g.K - 1) / g.K;  // k_first - tap >= -(K - 1)
        const int c_hi = (k_last - tap) >= 0 ? (k_last - tap) / g.K : -1;
        int c = c_lo < 0 ? 0 : c_lo;
        while (c <= c_hi) {
          const int gg = c / g.cg;
          const int c_end = min(c_hi, (gg + 1) * g.cg - 1);
          bool inside = false;
          float ly = 0.f, lx = 0.f;
          int y0 = 0, x0 = 0;
          if (px_ok) {
            const float py = (float)(b.x + ti * g.dh) + offs[(2 * (gg * g.K + tap)) * kFsBN + p];
            const float px = (float)(b.y + tj * g.dw) + offs[(2 * (gg * g.K + tap) + 1) * kFsBN + p];
            inside = touches_image(py, px, g.h, g.w);
            if (inside) {
              const float fy = floorf(py), fx = floorf(px);
              y0 = (int)fy;
              x0 = (int)fx;
              ly = py - fy;
              lx = px - fx;
            }
          }
          for (int c8 = c; c8 <= c_end; c8 += 8) {
            float cv[8][4];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              cv[u][0] = cv[u][1] = cv[u][2] = cv[u][3] = 0.f;
              if (inside && c8 + u <= c_end) {
                const __nv_bfloat16* plane = ximg + (long long)(c8 + u) * g.hw;
                cv[u][0] = corner(plane, g, y0, x0);
                cv[u][1] = corner(plane, g, y0, x0 + 1);
                cv[u][2] = corner(plane, g, y0 + 1, x0);
                cv[u][3] = corner(plane, g, y0 + 1, x0 + 1);
              }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              if (c8 + u > c_end) break;
              const float v = inside ? blend4(ly, lx, cv[u][0], cv[u][1], cv[u][2], cv[u][3]) : 0.f;
              const int kl = (c8 + u) * g.K + tap - k_first;
              *reinterpret_cast<unsigned short*>(sb + kl * 128 + (((p >> 3) ^ (kl & 7)) << 4) + (p & 7) * 2) =
                  __bfloat16_as_ushort(__float2bfloat16_rn(v));
            }
          }
          c = c_end + 1;
        }
      }
      // rows past the reduction (last block): zeros
      for (int kl = k_last - k_first + 1 + sw; kl < kBK; kl += kFsSampleWarps)
#pragma unroll
        for (int h = 0; h < kH; ++h) {
          const int p = lane + 32 * h;
          *reinterpret_cast<unsigned short*>(sb + kl * 128 + (((p >> 3) ^ (kl & 7)) << 4) + (p & 7) * 2) = 0;
        }
      // the tile is read by the tensor cores (async proxy)
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[s]);
    }
    if (warp < 4) {
      // ------------------------------------------------------------ epilogue
      ok = __all_sync(0xffffffffu, ok && mbar_wait(done, 0));
      tc_fence_after();
      const int row = warp * 32 + lane;
      const int m = m0 + row;
      const uint32_t tbase = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < kFsBN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tbase + c * 32, r);
        if (!ok || nkb == 0 || m >= g.c_out) continue;
        const int n_first = n0 + c * 32;
        if (g.relu) relu32(r);
        store_y_row(a.y + ((long long)n * g.c_out + m) * g.howo + n_first, r, n_first, (int)g.howo);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"((uint32_t)C::kTmemCols)
                 : "memory");
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// bf16 tensor map, 128-byte swizzle, zero fill outside the tensor.
bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
              const cuuint64_t* strides, const cuuint32_t* box,
              CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, dt, (cuuint32_t)rank, const_cast<void*>(base), dims,
            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int gemm_sm_count();

// `grid` is the tile grid.  Without a cluster the launch is persistent: one
// CTA per resident slot (shared and tensor memory bound it), each taking
// tiles blockIdx.x, + gridDim.x, ... of the tile grid.
template <int KIND, int BN, int MH = 1, int NACC = 2>
cudaError_t launch(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& Cm,
                   const TcArgs& args, dim3 grid, cudaStream_t s, int cluster_y = 1) {
  using C = Cfg<KIND, BN, MH, NACC>;
  auto k = tc_gemm<KIND, BN, MH, NACC>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
  if (e != cudaSuccess) return e;
  TcArgs a = args;
  a.vgx = (int)grid.x;
  a.vgy = (int)grid.y;
  a.vgz = (int)grid.z;
  a.persistent = cluster_y == 1 ? 1 : 0;
  dim3 g = grid;
  if (a.persistent) {
    const long long tiles = (long long)grid.x * grid.y * grid.z;
    int per_sm = (int)((227 * 1024) / (C::kSmem + 1024));
    if (per_sm > 512 / C::kTmemCols) per_sm = 512 / C::kTmemCols;
    if (per_sm < 1) per_sm = 1;
    const long long cap = (long long)per_sm * gemm_sm_count();
    g = dim3((unsigned)(tiles < cap ? tiles : cap), 1, 1);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = g;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int nattr = 0;
  // every GEMM may start its prologue (barriers, tensor memory) while its
  // predecessor finishes: FWD and GCOL wait for it before touching global
  // memory, GW (which reads nothing K4 writes) before it exits
  attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[nattr].val.programmaticStreamSerializationAllowed = 1;
  ++nattr;
  if (cluster_y > 1) {
    attr[nattr].id = cudaLaunchAttributeClusterDimension;
    attr[nattr].val.clusterDim.x = 1;
    attr[nattr].val.clusterDim.y = (unsigned)cluster_y;
    attr[nattr].val.clusterDim.z = 1;
    ++nattr;
  }
  cfg.attrs = attr;
  cfg.numAttrs = nattr;
  e = cudaLaunchKernelEx(&cfg, k, A, B, Cm, a);
  note_launches(1);
  return e;
}

// column buffer as a 3-D tensor {pixel (true extent), image, row}
bool col_map(CUtensorMap* m, const void* col, const Geom& g, const ColLayout& L, cuuint32_t box_rows) {
  const cuuint64_t dims[3] = {(cuuint64_t)g.howo, (cuuint64_t)g.n, (cuuint64_t)g.kdim};
  const cuuint64_t strides[2] = {(cuuint64_t)L.img * 2, (cuuint64_t)L.row * 2};
  const cuuint32_t box[3] = {64, 1, box_rows};
  return make_map(m, col, 3, dims, strides, box);
}

// grad_y as a 3-D tensor {pixel, channel, image}
// gcol (bf16) as the store target of the GCOL epilogue: boxes of 64 pixels x
// 32 rows of one image
bool gcol_map(CUtensorMap* m, const void* gcol, const Geom& g, const ColLayout& L) {
  const cuuint64_t dims[3] = {(cuuint64_t)g.howo, (cuuint64_t)g.n, (cuuint64_t)g.kdim};
  const cuuint64_t strides[2] = {(cuuint64_t)L.img * 2, (cuuint64_t)L.row * 2};
  const cuuint32_t box[3] = {64, 1, 32};
  return make_map(m, gcol, 3, dims, strides, box);
}

bool gy_map(CUtensorMap* m, const void* gy, const Geom& g, cuuint32_t box_ch) {
  const cuuint64_t dims[3] = {(cuuint64_t)g.howo, (cuuint64_t)g.c_out, (cuuint64_t)g.n};
  const cuuint64_t strides[2] = {(cuuint64_t)g.howo * 2, (cuuint64_t)g.c_out * g.howo * 2};
  const cuuint32_t box[3] = {64, box_ch, 1};
  return make_map(m, gy, 3, dims, strides, box);
}

// main weights as a 2-D tensor {kdim, c_out}
bool w_map(CUtensorMap* m, const void* w, const Geom& g, cuuint32_t box0, cuuint32_t box1) {
  const cuuint64_t dims[2] = {(cuuint64_t)g.kdim, (cuuint64_t)g.c_out};
  const cuuint64_t strides[1] = {(cuuint64_t)g.kdim * 2};
  const cuuint32_t box[2] = {box0, box1};
  return make_map(m, w, 2, dims, strides, box);
}

int gemm_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return 152;
  return sms;
}

int pick_fwd_bn(const Geom& g) {
  const long long tiles128 = ceil_div_ll(g.howo, 128) * ceil_div_ll(g.c_out, kBM) * g.n;
  return tiles128 >= 148 ? 128 : 64;
}

}  // namespace

// The tensor-core path needs 16-byte aligned rows for every tensor map.
bool tc_gemm_supported(const Geom& g) {
  return g.kdim % 8 == 0 && g.howo % 8 == 0 && encode_fn() != nullptr;
}

cudaError_t launch_gemm_fwd_tc(const GemmArgs& ga, cudaStream_t s) {
  const Geom& g = ga.g;
  CUtensorMap A, B;
  if (!w_map(&A, ga.w, g, 64, 128)) return cudaErrorInvalidValue;
  if (!col_map(&B, ga.col, g, ga.col_layout, 64)) return cudaErrorInvalidValue;
  TcArgs a{};
  a.c_out = g.c_out;
  a.kdim = g.kdim;
  a.howo = (int)g.howo;
  a.nimg = g.n;
  a.kb_total = (int)ceil_div_ll(g.kdim, kBK);
  a.out = ga.y;
  a.relu = g.relu;
  const int bn = pick_fwd_bn(g);
  const long long tiles = ceil_div_ll(g.howo, bn) * ceil_div_ll(g.c_out, kBM) * g.n;
  // fewer output tiles than SMs and a long reduction: split the k-blocks over
  // a 2-CTA cluster (measured: a gain from 36 k-blocks, a loss at 18)
  a.fwd_split = (bn == 64 && tiles < 152 && a.kb_total >= 24) ? 2 : 1;
  dim3 grid((unsigned)ceil_div_ll(g.howo, bn), (unsigned)(ceil_div_ll(g.c_out, kBM) * a.fwd_split),
            (unsigned)g.n);
  return bn == 128 ? launch<FWD, 128>(A, B, A, a, grid, s)
                   : launch<FWD, 64>(A, B, A, a, grid, s, a.fwd_split);
}

cudaError_t launch_gemm_gcol_tc(const GemmArgs& ga, cudaStream_t s) {
  const Geom& g = ga.g;
  CUtensorMap A, B, Cm;
  if (!w_map(&A, ga.w, g, 64, 64)) return cudaErrorInvalidValue;
  if (!gy_map(&B, ga.gy, g, 64)) return cudaErrorInvalidValue;
  if (!gcol_map(&Cm, ga.gcol, g, ga.gcol_layout)) return cudaErrorInvalidValue;
  TcArgs a{};
  a.c_out = g.c_out;
  a.kdim = g.kdim;
  a.howo = (int)g.howo;
  a.nimg = g.n;
  a.kb_total = (int)ceil_div_ll(g.c_out, kBK);
  a.out = ga.gcol;
  a.out_row = ga.gcol_layout.row;
  a.out_img = ga.gcol_layout.img;
  a.zero = ga.zero;
  a.gmax = ga.gmax;
  dim3 grid((unsigned)ceil_div_ll(g.howo, 128), (unsigned)ceil_div_ll(g.kdim, kBM), (unsigned)g.n);
  return launch<GCOL, 128>(A, B, Cm, a, grid, s);
}

cudaError_t launch_gemm_gw_tc(const GemmArgs& ga, cudaStream_t s) {
  const Geom& g = ga.g;
  CUtensorMap A, B;
  if (!gy_map(&A, ga.gy, g, 128)) return cudaErrorInvalidValue;
  if (!col_map(&B, ga.col, g, ga.col_layout, 128)) return cudaErrorInvalidValue;
  TcArgs a{};
  if (ga.gwo_img) {
    if ((ga.gwo_count & 3) || (reinterpret_cast<uintptr_t>(ga.gwo_img) & 15))
      return cudaErrorInvalidValue;
    a.gwo_img = ga.gwo_img;
    a.gw_off = ga.gw_off;
    a.gwo_count = ga.gwo_count;
    a.gwo_nimg = g.n;
    a.gwo_m = g.M;
    a.gwo_cin = g.c_in;
    a.gwo_k = g.K;
  }
  a.c_out = g.c_out;
  a.kdim = g.kdim;
  a.howo = (int)g.howo;
  a.nimg = g.n;
  a.qblocks = (int)ceil_div_ll(g.howo, kBK);
  a.kb_total = a.qblocks * g.n;
  a.out = ga.gw;
  const long long tiles = ceil_div_ll(g.kdim, 128) * ceil_div_ll(g.c_out, kBM);
  // about one CTA per SM: more splits only add float4 atomics on grad_W
  long long splits = ceil_div_ll(152, tiles);
  if (splits > a.kb_total) splits = a.kb_total;
  if (splits < 1) splits = 1;
  a.kb_per_split = (int)ceil_div_ll(a.kb_total, splits);
  splits = ceil_div_ll(a.kb_total, a.kb_per_split);
  dim3 grid((unsigned)ceil_div_ll(g.kdim, 128), (unsigned)ceil_div_ll(g.c_out, kBM), (unsigned)splits);
  return launch<GW, 128>(A, B, A, a, grid, s);
}

// pixel-major deformed map (or its gradient) as a 3-D tensor {(tap, channel), pixel, image}
bool colc_map(CUtensorMap* m, const void* col, const Geom& g, cuuint32_t box_px,
              cuuint32_t box_r = 64) {
  const cuuint64_t dims[3] = {(cuuint64_t)g.kdim, (cuuint64_t)g.howo, (cuuint64_t)g.n};
  const cuuint64_t strides[2] = {(cuuint64_t)g.kdim * 2, (cuuint64_t)g.howo * g.kdim * 2};
  const cuuint32_t box[3] = {box_r, box_px, 1};
  return make_map(m, col, 3, dims, strides, box);
}

cudaError_t launch_gemm_fwd_cl(const GemmArgs& ga, cudaStream_t s) {
  const Geom& g = ga.g;
  const int bn = pick_fwd_bn(g);
  CUtensorMap A, B;
  if (!w_map(&A, ga.w, g, 64, 128)) return cudaErrorInvalidValue;
  if (!colc_map(&B, ga.col, g, (cuuint32_t)bn)) return cudaErrorInvalidValue;
  TcArgs a{};
  a.c_out = g.c_out;
  a.kdim = g.kdim;
  a.howo = (int)g.howo;
  a.nimg = g.n;
  a.kb_total = (int)ceil_div_ll(g.kdim, kBK);
  a.out = ga.y;
  a.relu = g.relu;
  if (bn == 128 && g.c_out > kBM) {
    // all output channels of a pixel tile in one CTA (two halves): the map is
    // read once.  When 192-pixel tiles over the flat pixel index of all
    // images fit in one wave, those (one accumulator: 2 x 256 tensor-memory
    // columns; per k-block 56 KB filled for 6.3 MFLOP; a 32-pixel chunk of
    // the epilogue crosses at most one image boundary); else 96-pixel tiles
    // per image
    const long long total = (long long)g.n * g.howo;
    const long long flat_tiles = ceil_div_ll(total, 192) * ceil_div_ll(g.c_out, 2 * kBM);
    a.fwd_split = 1;
    if (flat_tiles <= gemm_sm_count() && total < INT_MAX && g.howo >= 32) {
      CUtensorMap Bf;
      const cuuint64_t dims[2] = {(cuuint64_t)g.kdim, (cuuint64_t)total};
      const cuuint64_t strides[1] = {(cuuint64_t)g.kdim * 2};
      const cuuint32_t box[2] = {64, 192};
      if (!make_map(&Bf, ga.col, 2, dims, strides, box)) return cudaErrorInvalidValue;
      a.flat = 1;
      dim3 grid((unsigned)ceil_div_ll(total, 192), (unsigned)ceil_div_ll(g.c_out, 2 * kBM), 1);
      return launch<FWDC, 192, 2, 1>(A, Bf, A, a, grid, s);
    }
    CUtensorMap B96;
    if (!colc_map(&B96, ga.col, g, 96)) return cudaErrorInvalidValue;
    dim3 grid((unsigned)ceil_div_ll(g.howo, 96), (unsigned)ceil_div_ll(g.c_out, 2 * kBM), (unsigned)g.n);
    return launch<FWDC, 96, 2>(A, B96, A, a, grid, s);
  }
  const long long tiles = ceil_div_ll(g.howo, bn) * ceil_div_ll(g.c_out, kBM) * g.n;
  a.fwd_split = (bn == 64 && tiles < 152 && a.kb_total >= 24) ? 2 : 1;
  dim3 grid((unsigned)ceil_div_ll(g.howo, bn), (unsigned)(ceil_div_ll(g.c_out, kBM) * a.fwd_split),
            (unsigned)g.n);
  return bn == 128 ? launch<FWDC, 128>(A, B, A, a, grid, s)
                   : launch<FWDC, 64>(A, B, A, a, grid, s, a.fwd_split);
}

cudaError_t launch_gemm_gcol_cl(const GemmArgs& ga, cudaStream_t s) {
  const Geom& g = ga.g;
  CUtensorMap A, B, Cm;
  if (!gy_map(&A, ga.gy, g, 64)) return cudaErrorInvalidValue;
  if (!w_map(&B, ga.w, g, 64, 64)) return cudaErrorInvalidValue;
  if (!colc_map(&Cm, ga.gcol, g, 32)) return cudaErrorInvalidValue;
  TcArgs a{};
  a.c_out = g.c_out;
  a.kdim = g.kdim;
  a.howo = (int)g.howo;
  a.nimg = g.n;
  a.kb_total = (int)ceil_div_ll(g.c_out, kBK);
  a.out = ga.gcol;
  a.zero = ga.zero;
  a.gmax = nullptr;
  if (g.kdim % 256 == 0) {
    // 256-column tiles: the grad_y tile (A) serves twice the columns
    dim3 grid((unsigned)(g.kdim / 256), (unsigned)ceil_div_ll(g.howo, kBM), (unsigned)g.n);
    return launch<GCOLC, 256>(A, B, Cm, a, grid, s);
  }
  dim3 grid((unsigned)ceil_div_ll(g.kdim, 128), (unsigned)ceil_div_ll(g.howo, kBM), (unsigned)g.n);
  return launch<GCOLC, 128>(A, B, Cm, a, grid, s);
}

cudaError_t launch_gemm_gw_cl(const GemmArgs& ga, cudaStream_t s) {
  const Geom& g = ga.g;
  CUtensorMap A, B;
  if (!gy_map(&A, ga.gy, g, 128)) return cudaErrorInvalidValue;
  if (!colc_map(&B, ga.col, g, 64)) return cudaErrorInvalidValue;
  TcArgs a{};
  if (ga.gwo_img) {
    if ((ga.gwo_count & 3) || (reinterpret_cast<uintptr_t>(ga.gwo_img) & 15))
      return cudaErrorInvalidValue;
    a.gwo_img = ga.gwo_img;
    a.gw_off = ga.gw_off;
    a.gwo_count = ga.gwo_count;
    a.gwo_nimg = g.n;
    a.gwo_m = g.M;
    a.gwo_cin = g.c_in;
    a.gwo_k = g.K;
  }
  a.c_out = g.c_out;
  a.kdim = g.kdim;
  a.howo = (int)g.howo;
  a.nimg = g.n;
  a.cin = ga.gw_perm ? 0 : g.c_in;
  a.ktaps = g.K;
  a.qblocks = (int)ceil_div_ll(g.howo, kBK);
  a.kb_total = a.qblocks * g.n;
  a.out = ga.gw_perm ? ga.gw_perm : ga.gw;
  // all output channels of a column tile in one CTA when C_out > 128 (two
  // halves: the map is read once); the pixels split over CTAs so that the
  // grid is one wave.  (256-column tiles with one accumulator fill fewer
  // bytes per flop but need twice the splits, and the float4 atomics that
  // add the splits into grad_W then cost more than they save.)
  const int mh = g.c_out > kBM ? 2 : 1;
  const int bn = 128;
  const long long tiles = ceil_div_ll(g.kdim, bn) * ceil_div_ll(g.c_out, kBM * mh);
  const int sms = gemm_sm_count();
  long long splits = sms / tiles;
  if (splits > a.kb_total) splits = a.kb_total;
  if (splits < 1) splits = 1;
  a.kb_per_split = (int)ceil_div_ll(a.kb_total, splits);
  splits = ceil_div_ll(a.kb_total, a.kb_per_split);
  dim3 grid((unsigned)ceil_div_ll(g.kdim, bn), (unsigned)ceil_div_ll(g.c_out, kBM * mh), (unsigned)splits);
  return mh == 2 ? launch<GWC, 128, 2>(A, B, A, a, grid, s) : launch<GWC, 128>(A, B, A, a, grid, s);
}

bool fwd_sampled_supported(const Geom& g) {
  return tc_gemm_supported(g) && fs_smem_bytes(g.M) <= 227 * 1024;
}

cudaError_t launch_fwd_sampled_tc(const Geom& g, const void* x, const void* w, const float* off,
                                  void* y, cudaStream_t s) {
  CUtensorMap A;
  if (!w_map(&A, w, g, 64, 128)) return cudaErrorInvalidValue;
  FsArgs a{};
  a.g = g;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.off = off;
  a.y = static_cast<__nv_bfloat16*>(y);
  a.kb_total = (int)ceil_div_ll(g.kdim, kBK);
  const size_t smem = fs_smem_bytes(g.M);
  cudaError_t e = cudaFuncSetAttribute(tc_fwd_sampled, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ceil_div_ll(g.howo, kFsBN), (unsigned)ceil_div_ll(g.c_out, kBM), (unsigned)g.n);
  cfg.blockDim = dim3(kFsThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, tc_fwd_sampled, A, a);
  note_launches(1);
  return e;
}

}  // namespace dc

namespace dc {
namespace {
// One thread waits, for at most `spins` polls, on an mbarrier that nothing
// arrives on; on expiry it raises the flag as every bounded wait of the
// library does.  No copy or tensor-memory allocation is outstanding.
__global__ void selftest_wait_kernel(unsigned int spins) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  for (unsigned int i = 0; i < spins; ++i)
    if (mbar_try_wait(&bar, 0)) return;
  atomicOr(&g_dc_device_error, 1u);
}
}  // namespace
}  // namespace dc

extern "C" dc_status dc_selftest_wait_timeout(unsigned int spins, void* stream) {
  if (spins == 0 || spins > (1u << 20)) return DC_ERR_INVALID_ARG;
  dc::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(spins);
  dc::note_launches(1);
  return cudaGetLastError() == cudaSuccess ? DC_OK : DC_ERR_CUDA;
}

// Reads (and optionally clears) the flag bounded device waits raise on expiry.
// The channels-last kernels and the float32 tensor-core GEMMs keep their own
// flags (cl_read_error, cl3_read_error, k4cl_read_error, tf32_read_error:
// 2 = unreadable).
extern "C" dc_status dc_device_error(int clear) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, dc::g_dc_device_error, sizeof(v)) != cudaSuccess) return DC_ERR_CUDA;
  if (clear && v) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(dc::g_dc_device_error, &zero, sizeof(zero)) != cudaSuccess)
      return DC_ERR_CUDA;
  }
  const unsigned int c = dc::cl_read_error(clear);
  const unsigned int c3 = dc::cl3_read_error(clear);
  const unsigned int c4 = dc::k4cl_read_error(clear);
  const unsigned int t = dc::tf32_read_error(clear);
  if (c == 2u || c3 == 2u || c4 == 2u || t == 2u) return DC_ERR_CUDA;
  return (v || c || c3 || c4 || t) ? DC_ERR_TIMEOUT : DC_OK;
}
