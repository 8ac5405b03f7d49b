// EvoFusion upstream stack on sm_103a: LayerNorm of the pair representation
// fused with the bias-free linear projection into q, k, v, g and the pair
// bias of triangle attention.
//
// MegaFold technical summary, "Methodik" section 3 "EvoFusion" (Umfang,
// Mechanismus): layer normalisation and the linear projections after it are
// restructured so that the normalised N x N x C tensor is never written to
// HBM between them.  Here each 128-row tile of z is normalised in shared
// memory, in place, and fed from there to the tensor core.
//
//   y[r, :]   = (z[r, :] - mean) / sqrt(var + eps) * gamma + beta     (r = (b, i, j))
//   out[r, o] = sum_c bf16(y[r, c]) * w[o, c]
//   q | k | v | g = out[r, 0:HD] | [HD:2HD] | [2HD:3HD] | [3HD:4HD]  ([B,N,N,H,D])
//   pair_bias[b, h, i, j] = out[r, 4HD + h]                           ([B,H,N,N])
//
// Persistent: one CTA per SM walks the 128-row tiles of z.  The 4*HD = 512
// q/k/v/g rows of w (128 KB, bf16) stay in shared memory for the whole
// kernel; the H pair-bias rows (fp32) and gamma/beta too.
//
// Warp roles (384 threads):
//   warp 0       TMA producer: w once, then z tiles into a 2-stage ring
//   warp 1       MMA issuer: out[:, 0:256] and out[:, 256:512] of a tile as two
//                M128 N256 products (K = C = 128) into the 512 columns of
//                tensor memory
//   warps 4-7    LayerNorm warpgroup: thread = row; normalises its row in place
//                (bf16, in the swizzled layout the MMA reads) and computes its
//                H pair-bias outputs with fp32 FMAs
//   warps 8-11   epilogue warpgroup: thread = TMEM lane = row; tensor memory ->
//                bf16 -> a 4 KB staging buffer per warp (32 rows x 128 B, in
//                the 128-byte swizzle) -> one TMA tensor store per chunk.  (A
//                thread storing its own row would touch 32 rows per store
//                instruction and saturate the load/store unit that the
//                LayerNorm warps share.)
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "layout.cuh"
#include "sm103.h"
#include "tmap.h"

namespace evo {
namespace {

struct FusionCfg {
  static constexpr int C = 128;        // channels of the pair representation
  static constexpr int HD = 128;       // H * D
  static constexpr int NOUT = 4 * HD;  // q, k, v, g columns (tensor core)
  static constexpr int HMAX = 8;       // pair-bias heads (CUDA cores)
  static constexpr int BM = 128;       // rows per tile
  static constexpr int NZ = 2;         // z stages
  static constexpr uint32_t HALF = 128 * 128;        // 128 rows x 64 channels bf16 (one box)
  static constexpr uint32_t ZTILE = 2 * HALF;        // a z tile: two 64-channel halves
  static constexpr uint32_t WHALF = NOUT * 128;      // 512 rows x 64 channels bf16
  // shared memory (offsets from a 1024-aligned base)
  static constexpr uint32_t OFF_W = 0;                       // [2 halves][512 rows][128 B]
  static constexpr uint32_t OFF_Z = OFF_W + 2 * WHALF;       // NZ x [2 halves][128 rows][128 B]
  static constexpr uint32_t OFF_WB = OFF_Z + NZ * ZTILE;     // [HMAX][C] fp32
  static constexpr uint32_t OFF_GB = OFF_WB + HMAX * C * 4;  // gamma[C], beta[C] fp32
  static constexpr uint32_t OFF_STAGE = OFF_GB + 2 * C * 4;  // 4 warps x 32 rows x 128 B
  static constexpr uint32_t SMEM = OFF_STAGE + 4 * 32 * 128;
  static constexpr uint32_t SMEM_ALLOC = SMEM + 1024;
  static constexpr int THREADS = 384;
  static constexpr int LAUNCH_REGS = 168, REGS_LOW = 64, REGS_LN = 224, REGS_EPI = 216;
  static_assert(REGS_LOW + REGS_LN + REGS_EPI <= 3 * LAUNCH_REGS, "register split");
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory");
};

struct FusionParams {
  int64_t rows;          // B * N * N
  int N, H, n_tiles;
  const __nv_bfloat16* w;  // [4HD + H, C]
  const float* gamma;
  const float* beta;
  float eps;
  __nv_bfloat16 *q, *k, *v, *g;  // [rows, HD]
  __nv_bfloat16* bias;            // [B, H, N, N]
  WaitCfg wc;
};

__global__ void __launch_bounds__(384, 1)
    evoattn_ln_proj_kernel(const __grid_constant__ CUtensorMap tm_z,
                           const __grid_constant__ CUtensorMap tm_w,
                           const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ CUtensorMap tm_g, const FusionParams p) {
  using C = FusionCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bar_w, bar_z_full[C::NZ], bar_z_empty[C::NZ], bar_y_ready[C::NZ],
      bar_mma_done[2], bar_tmem_free[2], bar_drain, bar_never;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int n_my = (p.n_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_w, 1);
    for (int i = 0; i < C::NZ; ++i) {
      mbar_init(&bar_z_full[i], 1);
      mbar_init(&bar_z_empty[i], 1);     // the tile's MMAs have read it
      mbar_init(&bar_y_ready[i], 128);   // every row normalised
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_mma_done[i], 1);
      mbar_init(&bar_tmem_free[i], 128);  // the epilogue has read the half's outputs
    }
    mbar_init(&bar_drain, 1);
    mbar_init(&bar_never, 1);            // nothing arrives: the stall test waits on it
    fence_barrier_init();
  }
  // the pair-bias rows of w (fp32), gamma and beta into shared memory
  {
    float* wb = reinterpret_cast<float*>(smem + C::OFF_WB);
    for (int i = threadIdx.x; i < p.H * C::C; i += C::THREADS)
      wb[i] = __bfloat162float(p.w[(int64_t)C::NOUT * C::C + i]);
    float* gb = reinterpret_cast<float*>(smem + C::OFF_GB);
    for (int i = threadIdx.x; i < C::C; i += C::THREADS) {
      gb[i] = p.gamma[i];
      gb[C::C + i] = p.beta[i];
    }
  }
  if (warp == 1) tmem_alloc(&tmem_slot, 512);
  if (warp == 0 && lane == 0) { tma_prefetch_desc(&tm_z); tma_prefetch_desc(&tm_w); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort_p = &abort_flag;
  const WaitCtx wctx{abort_p, p.wc};
  auto teardown = [&]() {
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem, 512);
    }
    if (threadIdx.x == 0) report_abort(abort_p, p.wc);
  };

  if (warp < 4) {
    regs_dec<C::REGS_LOW>();
    if (warp == 0) {
      // ============================ producer =================================
      bool ok = true;
      int issued = 0;
      if (lane == 0) mbar_arrive_expect_tx(&bar_w, 2 * C::WHALF);
      __syncwarp();
      // w: [2 channel halves][512 rows], one 128-row box per lane 0..7
      if (lane < 8) {
        const int hf = lane & 1, rg = lane >> 1;
        tma_load_2d(smem + C::OFF_W + hf * C::WHALF + rg * C::HALF, &tm_w, &bar_w, hf * 64,
                    rg * 128);
      }
      for (int n = 0; n < n_my && ok; ++n) {
        const int st = n % C::NZ;
        if (n >= C::NZ) ok = mbar_wait(&bar_z_empty[st], ((n / C::NZ) - 1) & 1, wctx);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const int row0 = ((int)blockIdx.x + n * (int)gridDim.x) * C::BM;
        if (lane == 0) mbar_arrive_expect_tx(&bar_z_full[st], C::ZTILE);
        __syncwarp();
        const int l0 = (2 * n) & 31;
        if (lane == l0)
          tma_load_2d(smem + C::OFF_Z + st * C::ZTILE, &tm_z, &bar_z_full[st], 0, row0);
        if (lane == ((l0 + 1) & 31))
          tma_load_2d(smem + C::OFF_Z + st * C::ZTILE + C::HALF, &tm_z, &bar_z_full[st], 64,
                      row0);
        issued = n + 1;
      }
      if (lane == 0) {  // every copy already issued lands before the CTA may exit
        volatile int no_abort = 0;
        if (!ok)
          for (int i = max(0, issued - C::NZ); i < issued; ++i)
            mbar_wait(&bar_z_full[i % C::NZ], (i / C::NZ) & 1, &no_abort);
        mbar_wait(&bar_w, 0, &no_abort);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ============================ MMA issuer ===============================
      // A = normalised tile (K-major, 128-byte swizzle, two 64-channel halves
      // 16 KB apart); B = w rows (K-major, 512 rows per channel half, halves
      // 64 KB apart).  K step kk (16 channels) is half kk / 4, byte offset
      // 32 * (kk % 4) within the swizzled 128-byte rows.
      constexpr uint32_t id = idesc_bf16(128, 256, 0, 0);
      const uint64_t da0 = umma_desc(smem_u32(smem + C::OFF_Z), 16, 1024, kSw128);
      const uint64_t db0 = umma_desc(smem_u32(smem + C::OFF_W), 16, 1024, kSw128);
      bool ok = __all_sync(0xffffffffu, mbar_wait(&bar_w, 0, wctx));
      for (int n = 0; n < n_my && ok; ++n) {
        const int st = n % C::NZ;
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_y_ready[st], (n / C::NZ) & 1, wctx));
        if (!ok) break;
        const uint64_t da = da0 + ((uint32_t)(st * C::ZTILE) >> 4);
        // half nh (q, k or v, g) once the epilogue has read the previous
        // tile's outputs of that half
#pragma unroll
        for (int nh = 0; nh < 2; ++nh) {
          if (n > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bar_tmem_free[nh], (n - 1) & 1, wctx));
            if (!ok) break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t a = da + ((uint32_t)((kk >> 2) * C::HALF + (kk & 3) * 32) >> 4);
            const uint64_t b =
                db0 + ((uint32_t)((kk >> 2) * C::WHALF + nh * 256 * 128 + (kk & 3) * 32) >> 4);
            if (elect_one()) umma_ss(tmem + 256 * nh, a, b, id, kk > 0 ? 1u : 0u);
          }
          if (elect_one()) {
            if (nh == 1) umma_commit(&bar_z_empty[st]);
            umma_commit(&bar_mma_done[nh]);
          }
          __syncwarp();
        }
        if (!ok) break;
      }
      if (elect_one()) umma_commit(&bar_drain);
      __syncwarp();
      if (lane == 0) {
        volatile int no_abort = 0;
        mbar_wait(&bar_drain, 0, &no_abort);
      }
      __syncwarp();
    }
    teardown();
  } else if (warp < 8) {
    // ============================ LayerNorm ==================================
    regs_inc<C::REGS_LN>();
    const int m = threadIdx.x - 128;  // row within the tile
    const float* wb = reinterpret_cast<const float*>(smem + C::OFF_WB);
    const float* gam = reinterpret_cast<const float*>(smem + C::OFF_GB);
    const float* bet = gam + C::C;
    const int64_t nn = (int64_t)p.N * p.N;
    bool ok = true;
    if (p.wc.stall) ok = __all_sync(0xffffffffu, stall_wait(&bar_never, wctx));
    for (int n = 0; n < n_my && ok; ++n) {
      const int st = n % C::NZ;
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_z_full[st], (n / C::NZ) & 1, wctx));
      if (!ok) break;
      uint8_t* zt = smem + C::OFF_Z + st * C::ZTILE;
      // the row, channel c in 16-byte chunk c / 8 of half c / 64 (chunk index
      // XOR row % 8: the 128-byte swizzle)
      float x[C::C];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 u = *reinterpret_cast<const uint4*>(zt + hf * C::HALF + m * 128 +
                                                          ((c ^ (m & 7)) << 4));
          float* xx = x + hf * 64 + c * 8;
          xx[0] = bf16lo(u.x); xx[1] = bf16hi(u.x); xx[2] = bf16lo(u.y); xx[3] = bf16hi(u.y);
          xx[4] = bf16lo(u.z); xx[5] = bf16hi(u.z); xx[6] = bf16lo(u.w); xx[7] = bf16hi(u.w);
        }
      // mean, then the mean squared deviation (two passes over registers)
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
      for (int c = 0; c < C::C; c += 4) { s0 += x[c]; s1 += x[c + 1]; s2 += x[c + 2]; s3 += x[c + 3]; }
      const float mean = ((s0 + s1) + (s2 + s3)) * (1.0f / C::C);
      s0 = s1 = s2 = s3 = 0.f;
#pragma unroll
      for (int c = 0; c < C::C; c += 4) {
        const float d0 = x[c] - mean, d1 = x[c + 1] - mean, d2 = x[c + 2] - mean,
                    d3 = x[c + 3] - mean;
        s0 = fmaf(d0, d0, s0); s1 = fmaf(d1, d1, s1); s2 = fmaf(d2, d2, s2); s3 = fmaf(d3, d3, s3);
      }
      const float var = ((s0 + s1) + (s2 + s3)) * (1.0f / C::C);
      const float rstd = rsqrtf(var + p.eps);
      // y = (x - mean) * rstd * gamma + beta, rounded to bf16, written back in
      // place; the pair-bias dot products use the same rounded y
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int c0 = hf * 64 + c * 8;
          const float4 ga = *reinterpret_cast<const float4*>(gam + c0);
          const float4 gb = *reinterpret_cast<const float4*>(gam + c0 + 4);
          const float4 ba = *reinterpret_cast<const float4*>(bet + c0);
          const float4 bb = *reinterpret_cast<const float4*>(bet + c0 + 4);
          const float gv[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
          const float bv[8] = {ba.x, ba.y, ba.z, ba.w, bb.x, bb.y, bb.z, bb.w};
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float y0 = fmaf((x[c0 + 2 * e] - mean) * rstd, gv[2 * e], bv[2 * e]);
            const float y1 = fmaf((x[c0 + 2 * e + 1] - mean) * rstd, gv[2 * e + 1], bv[2 * e + 1]);
            pk[e] = pack_bf16(y0, y1);
            x[c0 + 2 * e] = bf16lo(pk[e]);
            x[c0 + 2 * e + 1] = bf16hi(pk[e]);
          }
          *reinterpret_cast<uint4*>(zt + hf * C::HALF + m * 128 + ((c ^ (m & 7)) << 4)) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      fence_proxy_async_smem();  // generic writes, read by the tensor core
      mbar_arrive(&bar_y_ready[st]);
      const int64_t row = (int64_t)((int)blockIdx.x + n * (int)gridDim.x) * C::BM + m;
      if (row < p.rows) {
        const int64_t bidx = row / nn, rem = row % nn;
        for (int h = 0; h < p.H; ++h) {
          const float* w = wb + h * C::C;
          float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
          for (int c = 0; c < C::C; c += 4) {
            const float4 w4 = *reinterpret_cast<const float4*>(w + c);
            a0 = fmaf(x[c], w4.x, a0); a1 = fmaf(x[c + 1], w4.y, a1);
            a2 = fmaf(x[c + 2], w4.z, a2); a3 = fmaf(x[c + 3], w4.w, a3);
          }
          p.bias[(bidx * p.H + h) * nn + rem] = __float2bfloat16_rn((a0 + a1) + (a2 + a3));
        }
      }
    }
    teardown();
  } else {
    // ============================ epilogue ===================================
    regs_inc<C::REGS_EPI>();
    const int quad = warp & 3;
    const int m = quad * 32 + lane;  // TMEM lane = row within the tile
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    const CUtensorMap* outs[4] = {&tm_q, &tm_k, &tm_v, &tm_g};
    bool ok = true;
    for (int n = 0; n < n_my && ok; ++n) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_mma_done[0], n & 1, wctx));
      if (!ok) break;
      tc_fence_after();
      const int row0 = ((int)blockIdx.x + n * (int)gridDim.x) * C::BM + quad * 32;
      // this warp's staging buffer: row r, 16-byte chunk c at chunk c ^ (r % 8)
      uint8_t* stg = smem + C::OFF_STAGE + quad * 4096;
      // each output: 128 columns in two chunks of 64 (128 bytes of a row)
#pragma unroll 1
      for (int o = 0; o < 4 && ok; ++o) {
        if (o == 2) {  // v and g: the second half of tensor memory
          ok = __all_sync(0xffffffffu, mbar_wait(&bar_mma_done[1], n & 1, wctx));
          if (!ok) break;
          tc_fence_after();
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t ra[32], rb[32];
          tmem_ld32(lane_base + 128 * o + 64 * hh, ra);
          tmem_ld32(lane_base + 128 * o + 64 * hh + 32, rb);
          // the previous chunk's bulk store has read the staging buffer
          if (lane == 0) tma_store_wait_read();
          __syncwarp();
          tmem_wait_ld();
          reg_fence32(ra);
          reg_fence32(rb);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t* src = c < 4 ? &ra[8 * c] : &rb[8 * (c - 4)];
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                make_uint4(pack_bf16(__uint_as_float(src[0]), __uint_as_float(src[1])),
                           pack_bf16(__uint_as_float(src[2]), __uint_as_float(src[3])),
                           pack_bf16(__uint_as_float(src[4]), __uint_as_float(src[5])),
                           pack_bf16(__uint_as_float(src[6]), __uint_as_float(src[7])));
          }
          // generic writes, read by the bulk copy (rows beyond the tensor are
          // dropped by the copy)
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) tma_store_2d(outs[o], stg, 64 * hh, row0);
          __syncwarp();
        }
        if (o == 1 || o == 3) {  // a half of tensor memory is read
          tc_fence_before();
          mbar_arrive(&bar_tmem_free[o >> 1]);
        }
      }
      if (!ok) break;
    }
    if (lane == 0) tma_store_wait_all();
    __syncwarp();
    teardown();
  }
}

}  // namespace

cudaError_t bf16_ln_proj(const void* z, const float* gamma, const float* beta, const void* w,
                         float eps, void* q, void* k, void* v, void* g, void* bias, int B, int N,
                         int H, const WaitCfg& wait, cudaStream_t st, bool* tmap_ok) {
  using C = FusionCfg;
  const uint64_t rows = (uint64_t)B * N * N;
  CUtensorMap tz, tw, tq, tk, tv, tg;
  const uint64_t zdims[2] = {(uint64_t)C::C, rows};
  const uint64_t zstr[1] = {(uint64_t)C::C * 2};
  const uint32_t box[2] = {64, 128};
  const uint64_t wdims[2] = {(uint64_t)C::C, (uint64_t)C::NOUT};
  // outputs [rows, HD]: one bulk store writes 32 rows x 64 columns
  const uint64_t odims[2] = {(uint64_t)C::HD, rows};
  const uint64_t ostr[1] = {(uint64_t)C::HD * 2};
  const uint32_t obox[2] = {64, 32};
  if (!make_tmap_bf16(&tz, z, 2, zdims, zstr, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16(&tw, w, 2, wdims, zstr, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16(&tq, q, 2, odims, ostr, obox, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16(&tk, k, 2, odims, ostr, obox, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16(&tv, v, 2, odims, ostr, obox, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16(&tg, g, 2, odims, ostr, obox, CU_TENSOR_MAP_SWIZZLE_128B)) {
    *tmap_ok = false;
    return cudaErrorInvalidValue;
  }
  FusionParams fp{};
  fp.rows = (int64_t)rows;
  fp.N = N;
  fp.H = H;
  const uint64_t tiles = (rows + C::BM - 1) / C::BM;
  if (tiles > 0x7FFFFFFFull) return cudaErrorInvalidConfiguration;
  fp.n_tiles = (int)tiles;
  fp.w = static_cast<const __nv_bfloat16*>(w);
  fp.gamma = gamma;
  fp.beta = beta;
  fp.eps = eps;
  fp.q = static_cast<__nv_bfloat16*>(q);
  fp.k = static_cast<__nv_bfloat16*>(k);
  fp.v = static_cast<__nv_bfloat16*>(v);
  fp.g = static_cast<__nv_bfloat16*>(g);
  fp.bias = static_cast<__nv_bfloat16*>(bias);
  fp.wc = launch_wait(wait);
  auto kern = evoattn_ln_proj_kernel;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  // the warpgroups' register split must fit the pool the CTA is launched with
  cudaFuncAttributes fa{};
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs < C::LAUNCH_REGS) return cudaErrorInvalidConfiguration;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)std::min<uint64_t>(tiles, (uint64_t)std::max(sms, 1));
  kern<<<grid, C::THREADS, C::SMEM_ALLOC, st>>>(tz, tw, tq, tk, tv, tg, fp);
  return cudaGetLastError();
}

}  // namespace evo
