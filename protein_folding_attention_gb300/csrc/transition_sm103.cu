// EvoFusion downstream stack on sm_103a: the output projection of the gated
// attention with its residual add, then the SwiGLU transition of the pair
// representation (LayerNorm -> two bias-free projections -> SwiGLU -> the
// bias-free projection back -> residual add), as one kernel.
//
// MegaFold technical summary, "Methodik" section 3 "EvoFusion" (Umfang,
// Mechanismus): layer normalisation, the linear projections and the SwiGLU
// activation are restructured so that no intermediate N x N tensor (the
// normalised z, the 2F projections, the F-wide activation) is written to
// HBM.  Per 128-row tile, the normalised rows and the activation stay in
// shared memory, the projections in tensor memory:
//
//   z1[r, :]  = z[r, :] + o[r, :] w_o^T      (fp32; without o, z1 = z)
//   y[r, :]   = bf16((z1[r, :] - mean) / sqrt(var + eps) * gamma + beta)
//   a = y w1[0:F]^T,  b = y w1[F:2F]^T                 (r = (b, i, j); F = 4C)
//   h[r, f]   = bf16(silu(a[r, f]) * b[r, f]),  silu(x) = x / (1 + e^-x)
//   out[r, :] = bf16(z1[r, :] + h[r, :] w2^T)
//
// Persistent: one CTA per SM walks the 128-row tiles.  The weights (384 KB)
// do not fit in shared memory: they stream from L2 in chunks of 32 hidden
// units (the 64 rows of w1 that make a and b of those units, 16 KB, and the
// 32 columns of w2, 8 KB) through a ring of 6 stages (4 with the output
// projection, whose o tile and 32 KB w_o also sit in shared memory), every
// CTA reading the same 384 KB per tile.  The output projection accumulates
// into the tile's out accumulator, so out = z + o w_o^T + h w2^T comes out
// of one accumulator and one rounding.  The A operands of both products (y and h) live in
// tensor memory, which keeps the N = 64 first product compute-bound (with
// A in shared memory it ran at half rate) and leaves shared memory to the
// weight ring.
//
// Warp roles (512 threads):
//   warp 0       TMA producer of the weight ring
//   warp 1       MMA issuer: per chunk, [a | b] (M128 N64, K = C, A = y from
//                tensor memory) into one of two 64-column buffers, then the
//                running out += h_chunk w2_chunk^T (M128 N128, K = 32, A = h
//                from tensor memory) into one of two 128-column accumulators
//                (one per tile in flight)
//   warp 2       TMA producer of the z tiles (two stages)
//   warp 3       TMA producer of w_o (once) and the o tiles (one stage); the
//                MMA issuer computes o w_o^T of the next tile in the middle
//                of the current one (M128 N128, K = 128, both from shared
//                memory)
//   warps 4-7    LayerNorm (thread = row = TMEM lane: z1 = z + o w_o^T, y into
//                tensor memory)
//                and the epilogue (z + out -> bf16, written over the z tile in
//                place, one TMA tensor store per warp and 64-column half)
//   warps 8-15   SwiGLU, two warpgroups of 16 hidden units of each chunk:
//                thread = TMEM lane = row; a and b out of tensor memory, h
//                back into it
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

template <bool HAS_O>
struct TransitionCfg {
  static constexpr int C = 128;     // channels of the pair representation
  static constexpr int F = 4 * C;   // hidden units of the transition
  static constexpr int FC = 32;     // hidden units per chunk
  static constexpr int NCH = F / FC;
  static constexpr int BM = 128;    // rows per tile
  static constexpr int NZ = 2;      // z stages
  static constexpr int NW = HAS_O ? 4 : 6;  // weight stages
  static constexpr uint32_t HALF = 128 * 128;          // 128 rows x 64 channels bf16
  static constexpr uint32_t ZTILE = 2 * HALF;          // [2 halves][128 rows][128 B]
  static constexpr uint32_t W1C = 2 * 64 * 128;        // [2 k-halves][64 rows][128 B]
  static constexpr uint32_t W2C = C * FC * 2;          // [128 rows][64 B]
  static constexpr uint32_t WST = W1C + W2C;
  // shared memory (offsets from a 1024-aligned base)
  static constexpr uint32_t OFF_Z = 0;
  static constexpr uint32_t OFF_W = OFF_Z + NZ * ZTILE;
  static constexpr uint32_t OFF_O = OFF_W + NW * WST;               // o tile (HAS_O)
  static constexpr uint32_t OFF_WO = OFF_O + (HAS_O ? ZTILE : 0);   // w_o (HAS_O)
  static constexpr uint32_t OFF_GB = OFF_WO + (HAS_O ? ZTILE : 0);  // gamma[C], beta[C] fp32
  static constexpr uint32_t SMEM = OFF_GB + 2 * C * 4;
  static constexpr uint32_t SMEM_ALLOC = SMEM + 1024;
  // tensor memory columns (lane = row of the tile)
  static constexpr uint32_t T_ACC = 0;    // 2 x 128: out accumulators (fp32)
  static constexpr uint32_t T_G = 256;    // 2 x 64: [a | b] of a chunk (fp32)
  static constexpr uint32_t T_Y = 384;    // 64: y, bf16 pairs (channels 2c, 2c+1)
  static constexpr uint32_t T_H = 448;    // 2 x 16: h of a chunk, bf16 pairs
  static constexpr int THREADS = 512;
  static constexpr int LAUNCH_REGS = 128, REGS_LOW = 80, REGS_LN = 192, REGS_SW = 120;
  static_assert(REGS_LOW + REGS_LN + 2 * REGS_SW <= 4 * LAUNCH_REGS, "register split");
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory");
  static_assert(OFF_W % 1024 == 0 && WST % 1024 == 0 && OFF_O % 1024 == 0 &&
                    OFF_WO % 1024 == 0,
                "alignment");
};

struct TransitionParams {
  int64_t rows;  // B * N * N
  int n_tiles;
  const float* gamma;
  const float* beta;
  float eps;
  WaitCfg wc;
};

template <bool HAS_O>
__global__ void __launch_bounds__(512, 1)
    evoattn_transition_kernel(const __grid_constant__ CUtensorMap tm_z,
                              const __grid_constant__ CUtensorMap tm_w1,
                              const __grid_constant__ CUtensorMap tm_w2,
                              const __grid_constant__ CUtensorMap tm_out,
                              const __grid_constant__ CUtensorMap tm_o,
                              const __grid_constant__ CUtensorMap tm_wo,
                              const TransitionParams p) {
  using C = TransitionCfg<HAS_O>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bar_z_full[C::NZ], bar_z_empty[C::NZ], bar_w_full[C::NW],
      bar_w_empty[C::NW], bar_y_ready, bar_y_free, bar_g_full[2], bar_g_free[2], bar_h_full[2],
      bar_h_free[2], bar_acc_full[2], bar_acc_free[2], bar_acc0[2], bar_o_full, bar_o_empty,
      bar_wo, bar_drain, bar_never;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int n_my = (p.n_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  const int n_chunks = n_my * C::NCH;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < C::NZ; ++i) {
      mbar_init(&bar_z_full[i], 1);
      mbar_init(&bar_z_empty[i], 4);  // each epilogue warp's stores have read its rows
    }
    for (int i = 0; i < C::NW; ++i) {
      mbar_init(&bar_w_full[i], 1);
      mbar_init(&bar_w_empty[i], 1);
    }
    mbar_init(&bar_y_ready, 128);
    mbar_init(&bar_y_free, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_g_full[i], 1);
      mbar_init(&bar_g_free[i], 256);  // both SwiGLU warpgroups have read a and b
      mbar_init(&bar_h_full[i], 256);
      mbar_init(&bar_h_free[i], 1);
      mbar_init(&bar_acc_full[i], 1);
      mbar_init(&bar_acc_free[i], 128);
      mbar_init(&bar_acc0[i], 1);  // o w_o^T of the tile is in its accumulator
    }
    mbar_init(&bar_o_full, 1);
    mbar_init(&bar_o_empty, 1);
    mbar_init(&bar_wo, 1);
    mbar_init(&bar_drain, 1);
    mbar_init(&bar_never, 1);  // nothing arrives: the stall test waits on it
    fence_barrier_init();
  }
  {
    float* gb = reinterpret_cast<float*>(smem + C::OFF_GB);
    for (int i = threadIdx.x; i < C::C; i += C::THREADS) {
      gb[i] = p.gamma[i];
      gb[C::C + i] = p.beta[i];
    }
  }
  if (warp == 1) tmem_alloc(&tmem_slot, 512);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w1); tma_prefetch_desc(&tm_w2);
    tma_prefetch_desc(&tm_z); tma_prefetch_desc(&tm_out);
    if (HAS_O) { tma_prefetch_desc(&tm_o); tma_prefetch_desc(&tm_wo); }
  }
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
  auto tile_row0 = [&](int n) { return ((int)blockIdx.x + n * (int)gridDim.x) * C::BM; };

  if (warp < 4) {
    regs_dec<C::REGS_LOW>();
    if (warp == 0) {
      // ======================= weight producer ===============================
      // chunk q (hidden units 32 q .. 32 q + 31): w1 rows 32 q.. (a) and
      // F + 32 q.. (b), each channel half a 32-row box, to rows 0-31 and 32-63
      // of the stage's two k-halves; w2 columns 32 q.. as one 128-row box
      bool ok = true;
      int issued = 0;
      for (int gc = 0; gc < n_chunks && ok; ++gc) {
        const int st = gc % C::NW, q = gc % C::NCH;
        if (gc >= C::NW) ok = mbar_wait(&bar_w_empty[st], ((gc / C::NW) - 1) & 1, wctx);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        uint8_t* ws = smem + C::OFF_W + st * C::WST;
        if (lane == 0) mbar_arrive_expect_tx(&bar_w_full[st], C::WST);
        __syncwarp();
        const int l0 = (5 * gc) & 31;
        const int me = (lane - l0) & 31;  // this lane's copy, if < 5
        if (me < 4) {
          const int kh = me & 1, ab = me >> 1;
          tma_load_2d(ws + kh * (C::W1C / 2) + ab * 4096, &tm_w1, &bar_w_full[st], kh * 64,
                      ab * C::F + q * C::FC);
        } else if (me == 4) {
          tma_load_2d(ws + C::W1C, &tm_w2, &bar_w_full[st], q * C::FC, 0);
        }
        issued = gc + 1;
      }
      if (lane == 0 && !ok) {  // every copy already issued lands before the CTA may exit
        volatile int no_abort = 0;
        for (int i = max(0, issued - C::NW); i < issued; ++i)
          mbar_wait(&bar_w_full[i % C::NW], (i / C::NW) & 1, &no_abort);
      }
      __syncwarp();
    } else if (warp == 2) {
      // ========================== z producer =================================
      bool ok = true;
      int issued = 0;
      for (int n = 0; n < n_my && ok; ++n) {
        const int st = n % C::NZ;
        if (n >= C::NZ) ok = mbar_wait(&bar_z_empty[st], ((n / C::NZ) - 1) & 1, wctx);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        if (lane == 0) mbar_arrive_expect_tx(&bar_z_full[st], C::ZTILE);
        __syncwarp();
        if (lane < 2)
          tma_load_2d(smem + C::OFF_Z + st * C::ZTILE + lane * C::HALF, &tm_z, &bar_z_full[st],
                      lane * 64, tile_row0(n));
        issued = n + 1;
      }
      if (lane == 0 && !ok) {
        volatile int no_abort = 0;
        for (int i = max(0, issued - C::NZ); i < issued; ++i)
          mbar_wait(&bar_z_full[i % C::NZ], (i / C::NZ) & 1, &no_abort);
      }
      __syncwarp();
    } else if (warp == 3 && HAS_O) {
      // ===================== w_o and o tile producer =========================
      bool ok = true;
      int issued = 0;
      if (lane == 0) mbar_arrive_expect_tx(&bar_wo, C::ZTILE);
      __syncwarp();
      if (lane < 2)
        tma_load_2d(smem + C::OFF_WO + lane * C::HALF, &tm_wo, &bar_wo, lane * 64, 0);
      for (int n = 0; n < n_my && ok; ++n) {
        if (n >= 1) ok = mbar_wait(&bar_o_empty, (n - 1) & 1, wctx);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        if (lane == 0) mbar_arrive_expect_tx(&bar_o_full, C::ZTILE);
        __syncwarp();
        if (lane < 2)
          tma_load_2d(smem + C::OFF_O + lane * C::HALF, &tm_o, &bar_o_full, lane * 64,
                      tile_row0(n));
        issued = n + 1;
      }
      if (lane == 0) {
        volatile int no_abort = 0;
        if (!ok && issued > 0) mbar_wait(&bar_o_full, (issued - 1) & 1, &no_abort);
        mbar_wait(&bar_wo, 0, &no_abort);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ============================ MMA issuer ===============================
      // A operands from tensor memory: K step kk (16 bf16) is 8 columns.
      // The w1 chunk: K-major, 128-byte swizzle, channel halves 8 KB apart;
      // K step kk is half kk / 4 at byte 32 (kk % 4) of the rows.  The w2
      // chunk: K-major, 64-byte swizzle, one 64-byte row per output channel;
      // K step kk at byte 32 kk.
      constexpr uint32_t id1 = idesc_bf16(128, 64, 0, 0);
      constexpr uint32_t id2 = idesc_bf16(128, 128, 0, 0);
      const uint64_t dw0 = umma_desc(smem_u32(smem + C::OFF_W), 16, 1024, kSw128);
      const uint64_t dw2 = umma_desc(smem_u32(smem + C::OFF_W + C::W1C), 16, 512, kSw64);
      bool ok = true;
      // o w_o^T of tile n into its accumulator (A = o tile, B = w_o: K-major,
      // 128-byte swizzle, channel halves 16 KB apart), once the epilogue of
      // tile n - 2 has read that accumulator
      auto gemm0 = [&](int n) -> bool {
        const int ta = n & 1;
        if (!mbar_wait(&bar_o_full, n & 1, wctx)) return false;
        if (n >= 2 && !mbar_wait(&bar_acc_free[ta], ((n >> 1) - 1) & 1, wctx)) return false;
        tc_fence_after();
        const uint64_t da = umma_desc(smem_u32(smem + C::OFF_O), 16, 1024, kSw128);
        const uint64_t db = umma_desc(smem_u32(smem + C::OFF_WO), 16, 1024, kSw128);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (uint32_t)((kk >> 2) * C::HALF + (kk & 3) * 32) >> 4;
          if (elect_one()) umma_ss(tmem + C::T_ACC + 128 * ta, da + off, db + off, id2, kk > 0);
        }
        if (elect_one()) {
          umma_commit(&bar_o_empty);
          umma_commit(&bar_acc0[ta]);
        }
        __syncwarp();
        return true;
      };
      if (HAS_O) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_wo, 0, wctx));
        if (ok && n_my > 0) ok = __all_sync(0xffffffffu, gemm0(0));
      }
      // the second product of global chunk gc (out += h w2^T): its h is ready
      auto gemm2 = [&](int gc) -> bool {
        const int hb = gc & 1, st = gc % C::NW, q = gc % C::NCH, ta = (gc / C::NCH) & 1;
        if (!mbar_wait(&bar_h_full[hb], (gc >> 1) & 1, wctx)) return false;
        tc_fence_after();
        const uint64_t b = dw2 + ((uint32_t)(st * C::WST) >> 4);
#pragma unroll
        for (int kk = 0; kk < C::FC / 16; ++kk)
          if (elect_one())
            umma_ts(tmem + C::T_ACC + 128 * ta, tmem + C::T_H + 16 * hb + 8 * kk, b + 2 * kk,
                    id2, (HAS_O || q > 0 || kk > 0) ? 1u : 0u);
        if (elect_one()) {
          umma_commit(&bar_h_free[hb]);
          umma_commit(&bar_w_empty[st]);
          if (q == C::NCH - 1) umma_commit(&bar_acc_full[ta]);
        }
        __syncwarp();
        return true;
      };
      for (int n = 0; n < n_my && ok; ++n) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_y_ready, n & 1, wctx));
        for (int q = 0; q < C::NCH && ok; ++q) {
          const int gc = n * C::NCH + q, st = gc % C::NW, gb = gc & 1;
          ok = mbar_wait(&bar_w_full[st], (gc / C::NW) & 1, wctx);
          if (ok && gc >= 2) ok = mbar_wait(&bar_g_free[gb], ((gc >> 1) - 1) & 1, wctx);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          const uint64_t b0 = dw0 + ((uint32_t)(st * C::WST) >> 4);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t b = b0 + ((uint32_t)((kk >> 2) * (C::W1C / 2) + (kk & 3) * 32) >> 4);
            if (elect_one())
              umma_ts(tmem + C::T_G + 64 * gb, tmem + C::T_Y + 8 * kk, b, id1, kk > 0 ? 1u : 0u);
          }
          if (elect_one()) {
            umma_commit(&bar_g_full[gb]);
            if (q == C::NCH - 1) umma_commit(&bar_y_free);
          }
          __syncwarp();
          if (q > 0) {
            // without o, the second product of a tile's chunk 0 needs its
            // accumulator read out by the epilogue of the tile two back (with
            // o, the output projection waited for it)
            if (!HAS_O && q == 1 && n >= 2)
              ok = __all_sync(0xffffffffu,
                              mbar_wait(&bar_acc_free[n & 1], ((n >> 1) - 1) & 1, wctx));
            if (ok) ok = __all_sync(0xffffffffu, gemm2(gc - 1));
          }
          // the next tile's output projection, early enough for its
          // LayerNorm to be done when this tile's first products end
          if (HAS_O && ok && q == C::NCH / 2 && n + 1 < n_my)
            ok = __all_sync(0xffffffffu, gemm0(n + 1));
        }
        if (ok) ok = __all_sync(0xffffffffu, gemm2(n * C::NCH + C::NCH - 1));
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
    // ===================== LayerNorm and epilogue ============================
    regs_inc<C::REGS_LN>();
    const int quad = warp & 3;
    const int m = quad * 32 + lane;  // row within the tile = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    const float* gam = reinterpret_cast<const float*>(smem + C::OFF_GB);
    const float* bet = gam + C::C;
    bool ok = true;
    if (p.wc.stall) ok = __all_sync(0xffffffffu, stall_wait(&bar_never, wctx));
    // out = z + acc for tile n, written over the z rows, then stored
    auto epilogue = [&](int n) -> bool {
      const int st = n % C::NZ, ta = n & 1;
      if (!mbar_wait(&bar_acc_full[ta], (n >> 1) & 1, wctx)) return false;
      tc_fence_after();
      uint8_t* zt = smem + C::OFF_Z + st * C::ZTILE;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t ra[32], rb[32];
        tmem_ld32(lane_base + C::T_ACC + 128 * ta + 64 * hf, ra);
        tmem_ld32(lane_base + C::T_ACC + 128 * ta + 64 * hf + 32, rb);
        tmem_wait_ld();
        reg_fence32(ra);
        reg_fence32(rb);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t* acc = c < 4 ? &ra[8 * c] : &rb[8 * (c - 4)];
          uint4* zp = reinterpret_cast<uint4*>(zt + hf * C::HALF + m * 128 + ((c ^ (m & 7)) << 4));
          const uint4 u = *zp;
          const uint32_t zw[4] = {u.x, u.y, u.z, u.w};
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            o[e] = pack_bf16(bf16lo(zw[e]) + __uint_as_float(acc[2 * e]),
                             bf16hi(zw[e]) + __uint_as_float(acc[2 * e + 1]));
          *zp = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&bar_acc_free[ta]);
      // generic writes, read by the bulk copy (rows beyond the tensor are
      // dropped by the copy)
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int row0 = tile_row0(n) + quad * 32;
        tma_store_2d(&tm_out, zt + quad * 4096, 0, row0);
        tma_store_2d(&tm_out, zt + C::HALF + quad * 4096, 64, row0);
        tma_store_wait_read();  // the z stage may be reloaded once read
        mbar_arrive(&bar_z_empty[st]);
      }
      __syncwarp();
      return true;
    };
    for (int n = 0; n < n_my && ok; ++n) {
      const int st = n % C::NZ;
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_z_full[st], (n / C::NZ) & 1, wctx));
      if (!ok) break;
      const uint8_t* zt = smem + C::OFF_Z + st * C::ZTILE;
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
      if (HAS_O) {  // z1 = z + o w_o^T (fp32, from the tile's accumulator)
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_acc0[n & 1], (n >> 1) & 1, wctx));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t ra[32];
          tmem_ld32(lane_base + C::T_ACC + 128 * (n & 1) + 32 * c, ra);
          tmem_wait_ld();
          reg_fence32(ra);
#pragma unroll
          for (int e = 0; e < 32; ++e) x[32 * c + e] += __uint_as_float(ra[e]);
        }
      }
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
      // y may be overwritten once the previous tile's first products are done
      if (n > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_y_free, (n - 1) & 1, wctx));
        if (!ok) break;
        tc_fence_after();
      }
      // y as 64 columns of bf16 pairs: the A operand of the first product
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int c0 = hf * 64 + c * 8;
          const float4 ga = *reinterpret_cast<const float4*>(gam + c0);
          const float4 gb = *reinterpret_cast<const float4*>(gam + c0 + 4);
          const float4 ba = *reinterpret_cast<const float4*>(bet + c0);
          const float4 bb = *reinterpret_cast<const float4*>(bet + c0 + 4);
          const float gv[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
          const float bv[8] = {ba.x, ba.y, ba.z, ba.w, bb.x, bb.y, bb.z, bb.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            pk[4 * c + e] =
                pack_bf16(fmaf((x[c0 + 2 * e] - mean) * rstd, gv[2 * e], bv[2 * e]),
                          fmaf((x[c0 + 2 * e + 1] - mean) * rstd, gv[2 * e + 1], bv[2 * e + 1]));
        }
        tmem_st32(lane_base + C::T_Y + 32 * hf, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar_y_ready);
      // the previous tile's epilogue runs while this tile's chunks go through
      // the tensor core
      if (n > 0) ok = __all_sync(0xffffffffu, epilogue(n - 1));
    }
    if (ok && n_my > 0) ok = __all_sync(0xffffffffu, epilogue(n_my - 1));
    if (lane == 0) tma_store_wait_all();
    __syncwarp();
    teardown();
  } else {
    // ============================== SwiGLU ===================================
    regs_dec<C::REGS_SW>();
    const int wgi = (warp - 8) >> 2;  // 16 hidden units of each chunk
    const int quad = warp & 3;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    bool ok = true;
    for (int gc = 0; gc < n_chunks && ok; ++gc) {
      const int gb = gc & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_g_full[gb], (gc >> 1) & 1, wctx));
      if (!ok) break;
      tc_fence_after();
      uint32_t ra[16], rb[16];
      tmem_ld16(lane_base + C::T_G + 64 * gb + 16 * wgi, ra);       // a
      tmem_ld16(lane_base + C::T_G + 64 * gb + 32 + 16 * wgi, rb);  // b
      tmem_wait_ld();
      reg_fence16(ra);
      reg_fence16(rb);
      tc_fence_before();
      mbar_arrive(&bar_g_free[gb]);
      // silu(a) b = a sigmoid(a) b, sigmoid(a) = 1 / (1 + 2^(-a log2 e))
      constexpr float kLog2e = 1.4426950408889634f;
      uint32_t hp[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float a0 = __uint_as_float(ra[2 * e]), a1 = __uint_as_float(ra[2 * e + 1]);
        const float h0 = __fdividef(a0, 1.0f + ex2(-a0 * kLog2e)) * __uint_as_float(rb[2 * e]);
        const float h1 =
            __fdividef(a1, 1.0f + ex2(-a1 * kLog2e)) * __uint_as_float(rb[2 * e + 1]);
        hp[e] = pack_bf16(h0, h1);
      }
      // the h columns are free once the second product two chunks back is done
      if (gc >= 2) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_h_free[gb], ((gc >> 1) - 1) & 1, wctx));
        if (!ok) break;
        tc_fence_after();
      }
      tmem_st8(lane_base + C::T_H + 16 * gb + 8 * wgi, hp);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar_h_full[gb]);
    }
    teardown();
  }
}

}  // namespace

namespace {

template <bool HAS_O>
cudaError_t launch_transition(const CUtensorMap& tz, const CUtensorMap& tw1,
                              const CUtensorMap& tw2, const CUtensorMap& tout,
                              const CUtensorMap& to, const CUtensorMap& two,
                              const TransitionParams& tp, uint64_t tiles, cudaStream_t st) {
  using C = TransitionCfg<HAS_O>;
  auto kern = evoattn_transition_kernel<HAS_O>;
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
  kern<<<grid, C::THREADS, C::SMEM_ALLOC, st>>>(tz, tw1, tw2, tout, to, two, tp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t bf16_transition(const void* z, const void* o, const void* w_o, const float* gamma,
                            const float* beta, const void* w1, const void* w2, float eps,
                            void* out, int B, int N, const WaitCfg& wait, cudaStream_t st,
                            bool* tmap_ok) {
  using C = TransitionCfg<false>;
  const uint64_t rows = (uint64_t)B * N * N;
  CUtensorMap tz, tw1, tw2, tout, to, two;
  const uint64_t zdims[2] = {(uint64_t)C::C, rows};
  const uint64_t zstr[1] = {(uint64_t)C::C * 2};
  const uint32_t zbox[2] = {64, 128};
  const uint64_t w1dims[2] = {(uint64_t)C::C, (uint64_t)(2 * C::F)};
  const uint32_t w1box[2] = {64, 32};
  const uint64_t w2dims[2] = {(uint64_t)C::F, (uint64_t)C::C};
  const uint64_t w2str[1] = {(uint64_t)C::F * 2};
  const uint32_t w2box[2] = {(uint32_t)C::FC, (uint32_t)C::C};
  const uint32_t obox[2] = {64, 32};
  // o [rows, H*D = 128] and w_o [C, H*D]: 128-row boxes of 64 channels, like z
  const uint64_t wodims[2] = {(uint64_t)C::C, (uint64_t)C::C};
  if (!make_tmap_bf16(&tz, z, 2, zdims, zstr, zbox, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16(&tw1, w1, 2, w1dims, zstr, w1box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_bf16(&tw2, w2, 2, w2dims, w2str, w2box, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_tmap_bf16(&tout, out, 2, zdims, zstr, obox, CU_TENSOR_MAP_SWIZZLE_128B) ||
      (o && (!make_tmap_bf16(&to, o, 2, zdims, zstr, zbox, CU_TENSOR_MAP_SWIZZLE_128B) ||
             !make_tmap_bf16(&two, w_o, 2, wodims, zstr, zbox, CU_TENSOR_MAP_SWIZZLE_128B)))) {
    *tmap_ok = false;
    return cudaErrorInvalidValue;
  }
  TransitionParams tp{};
  tp.rows = (int64_t)rows;
  const uint64_t tiles = (rows + C::BM - 1) / C::BM;
  if (tiles > 0x7FFFFFFFull / C::NCH) return cudaErrorInvalidConfiguration;
  tp.n_tiles = (int)tiles;
  tp.gamma = gamma;
  tp.beta = beta;
  tp.eps = eps;
  tp.wc = launch_wait(wait);
  return o ? launch_transition<true>(tz, tw1, tw2, tout, to, two, tp, tiles, st)
           : launch_transition<false>(tz, tw1, tw2, tout, tz, tz, tp, tiles, st);
}

}  // namespace evo
