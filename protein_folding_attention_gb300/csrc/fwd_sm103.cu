// EvoAttention forward on sm_103a: TMA-fed tcgen05 MMAs with TMEM
// accumulators and an online softmax in registers.
//
// MegaFold technical summary, "Methodik" section 1 "EvoFlash-3D": the logits
// of one query tile against one key tile are produced in on-chip memory and
// folded into a running (max, sum) pair -- the online normalizer of softmax --
// so the B*S*H*N*N attention map never reaches HBM; the pair bias, broadcast
// over the S rows, is added to every logit tile.
//
// CTA = one (b, h, 128-row query tile jt) and a group of G consecutive rows s.
// The key tiles kt form the outer loop and the G rows the inner loop, so each
// 128x128 pair-bias tile is loaded into shared memory once and serves G rows.
//
// The pair bias is added by the tensor core.  Each logit tile accumulates
//   T = Q K^T + (c I) * bias,      c = sqrt(D) rounded to bf16,
// in tensor memory (I the 128x128 identity, so the second product has one
// nonzero term per sum and adds c * bias[j, k] exactly in fp32); the softmax
// then works on T / sqrt(D).  c is exact for D = 16 and 64; for D = 32 it is
// 5.65625 against sqrt(32) = 5.656854, a relative error of 1.1e-4 in the bias
// coefficient, twenty times below the bf16 rounding that P gets before the
// PV product.  The identity is never stored whole: reduction chunk kk (bias
// rows j' in [16kk, 16kk+16)) is the 128-row window, starting at row
// 112 - 16kk, of a 240 x 16 matrix Z whose only nonzeros are Z[112 + i][i] =
// c.  The MMA reads the bias tile in the layout the TMA delivers it: keys
// contiguous (starting node, MSA) as an MN-major operand, queries contiguous
// (the ending-node view) as a K-major operand, so neither is transposed.
//
// Warp roles (384 threads, three warpgroups):
//   warp 0      TMA producer: Q tiles, K/V tiles of each (kt, s) and the
//               additive key mask of that (s, kt)
//   warp 1      MMA issuer of T, every tile in order
//   warp 2      MMA issuer of O += P V (P read from tensor memory), every
//               tile in order
//   warp 3      TMA producer of the bias tile of each kt
//   warps 4-7   softmax warpgroup 0: rows s = 0, 2, ... of the group
//   warps 8-11  softmax warpgroup 1: rows s = 1, 3, ...
// A softmax thread owns one query row j (TMEM lane 32*(warp%4) + lane).
//
// Tensor memory (512 columns): three T buffers at 0, 128, 256 (fp32
// 128x128), used by tile i = kt*G + s in turn (buffer i % 3); the bf16 P of a
// tile overwrites the first 64 columns of its buffer.  O of row s at 384 +
// s*D (fp32 128xD).  With three buffers the T of a warpgroup's next tile is
// computed while the warpgroup still works on its current one.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "layout.cuh"
#include "sm103.h"
#include "tmap.h"

namespace evo {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct FwdCfg {
  static constexpr int BM = 128;                   // query rows per tile
  static constexpr int BN = 128;                   // keys per tile
  static constexpr int G = (D == 64) ? 2 : 4;      // rows s per CTA
  static constexpr int NS = (D == 64) ? 3 : 5;     // K/V pipeline stages
  static constexpr int NT = 3;                     // T buffers in tensor memory
  static constexpr uint32_t ROW = D * 2;           // bytes of one bf16 row
  static constexpr uint32_t ATOM = 8 * ROW;        // swizzle atom (8 rows)
  static constexpr Swizzle SW = D == 16 ? kSw32 : (D == 32 ? kSw64 : kSw128);
  static constexpr uint32_t TILE = 128 * ROW;      // one 128-row Q/K/V tile
  static constexpr uint32_t BIAS_TILE = 128 * 128 * 2;
  static constexpr uint32_t Z_BYTES = 240 * 32;    // identity windows, 32-byte rows
  // shared memory carve-up (offsets from a 1024-aligned base)
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + G * TILE;
  static constexpr uint32_t OFF_V = OFF_K + NS * TILE;
  static constexpr uint32_t OFF_BIAS = OFF_V + NS * TILE;       // 2 stages
  static constexpr uint32_t OFF_Z = OFF_BIAS + 2 * BIAS_TILE;
  static constexpr uint32_t OFF_MADD = OFF_Z + Z_BYTES;
  static constexpr uint32_t OFF_FLAG = OFF_MADD + NS * BN * 4;  // per stage: tile has masked keys
  static constexpr uint32_t SMEM = OFF_FLAG + NS * 16;
  static constexpr uint32_t SMEM_ALLOC = SMEM + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t TMEM_O = 384;
  static constexpr int THREADS = 384;
  // register split: launch 168/thread; the producer warpgroup drops to 104,
  // the softmax warpgroups rise to 192 (104*128 + 192*256 <= 168*384; the
  // split with no spills in either region)
  static constexpr int LAUNCH_REGS = 168, REGS_LOW = 104, REGS_HIGH = 192;
  static_assert(REGS_LOW * 128 + REGS_HIGH * 256 <= LAUNCH_REGS * THREADS, "register split");
  static_assert(NT * 128 <= TMEM_O && TMEM_O + G * D <= TMEM_COLS, "tensor memory overflow");
  static_assert(OFF_BIAS % 1024 == 0 && OFF_Z % 256 == 0, "operand alignment");
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory");
};

struct FwdParams {
  int B, S, H, N;
  int n_jt, n_kt, n_sg;
  const unsigned char* mask;
  int64_t msb, mss, msk;
  const __nv_bfloat16* gate;
  Strides5 g;
  __nv_bfloat16* out;
  Strides5 o;
  float* lse;
  WaitCfg wc;
};

template <int D, bool BIAS_K_CONTIG, bool HAS_GATE>
__global__ void __launch_bounds__(384, 1)
    evoattn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_bias, const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bar_q, bar_kv_full[C::NS], bar_kv_empty[C::NS], bar_bias_full[2],
      bar_bias_empty[2], bar_s_full[C::NT], bar_s_free[C::NT], bar_p_ready[C::NT],
      bar_o_done[C::G], bar_drain[2], bar_never;
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;

  // ---- tile coordinates -------------------------------------------------
  int idx = blockIdx.x;
  const int jt = idx % p.n_jt; idx /= p.n_jt;
  const int h = idx % p.H; idx /= p.H;
  const int sg = idx % p.n_sg;
  const int b = idx / p.n_sg;
  const int s0 = sg * C::G;
  const int g_eff = min(C::G, p.S - s0);
  const int nkt = p.n_kt;
  const int total = nkt * g_eff;
  const int n_wg = g_eff >= 2 ? 2 : 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_q, 1);
    for (int i = 0; i < C::NS; ++i) { mbar_init(&bar_kv_full[i], 1); mbar_init(&bar_kv_empty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_bias_full[i], 1);
      mbar_init(&bar_bias_empty[i], 1);  // after the last T of a kt
      mbar_init(&bar_drain[i], 1);
    }
    // T ready / P ready / buffer free, one of each per T buffer: the next
    // completion of a buffer's barrier needs the buffer's current tile to
    // have been consumed, so no waiter can fall two phases behind
    for (int i = 0; i < C::NT; ++i) {
      mbar_init(&bar_s_full[i], 1);
      mbar_init(&bar_p_ready[i], 128);  // the warpgroup owning the tile
      mbar_init(&bar_s_free[i], 1);
    }
    for (int i = 0; i < C::G; ++i) mbar_init(&bar_o_done[i], 1);
    mbar_init(&bar_never, 1);  // nothing arrives: the stall test waits on it
    fence_barrier_init();
  }
  // Z in the 32-byte-swizzled K-major layout the MMA reads: row r holds 16
  // bf16 values in two 16-byte chunks, stored swapped when bit 2 of r is set.
  {
    const uint32_t cb = __bfloat16_as_ushort(__float2bfloat16_rn(sqrtf((float)D)));
    uint32_t* z32 = reinterpret_cast<uint32_t*>(smem + C::OFF_Z);
    for (int i = threadIdx.x; i < (int)(C::Z_BYTES / 4); i += C::THREADS) {
      const int r = i >> 3, wd = i & 7;
      const int c0 = (((wd >> 2) ^ ((r >> 2) & 1)) << 3) + ((wd & 3) << 1);
      const int one = r - 112;  // column of this row's nonzero, if any
      z32[i] = one == c0 ? cb : (one == c0 + 1 ? cb << 16 : 0u);
    }
    fence_proxy_async_smem();  // generic writes, read by the tensor core
  }
  if (warp == 1) tmem_alloc(&tmem_base_slot, C::TMEM_COLS);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q); tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v); tma_prefetch_desc(&tm_bias);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_slot;
  volatile int* abort_p = &abort_flag;
  const WaitCtx wctx{abort_p, p.wc};

  // Every role ends here: all MMAs and TMEM traffic are done once every
  // thread has arrived, then the allocating warp frees the tensor memory.
  auto teardown = [&]() {
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem, C::TMEM_COLS);
    }
    if (threadIdx.x == 0) report_abort(abort_p, p.wc);
  };
  if (warp < 4) {
  // setmaxnreg is warpgroup-aligned: one instance for warps 0-3, one for 4-11
  regs_dec<C::REGS_LOW>();
  if (warp == 0) {
    // =================== TMA producer (whole warp) ========================
    // The copy engine serves the copies one thread issues in order, but
    // those of different threads concurrently; with 64-byte rows a single
    // issuing thread would cap the loads at ~10 bytes/clock.  Each box is
    // therefore issued by the next lane of the warp in turn (the whole warp
    // calls these helpers; lane 0 arms the barrier first).
    int rr = 0;
    if (lane == 0) mbar_arrive_expect_tx(&bar_q, g_eff * C::TILE);
    __syncwarp();
    if (lane < g_eff)
      tma_load_5d(smem + C::OFF_Q + lane * C::TILE, &tm_q, &bar_q, 0, jt * C::BM, h, s0 + lane, b);
    rr = g_eff;
    bool ok = true;
    int kv_issued = 0;
    // mask bytes of the next (kt, s) are loaded while the current is armed
    unsigned char pre_m[4];
    auto prefetch_mask = [&](int i) {
      if (i >= total || !p.mask) return;
      const int pkt = i / g_eff, ps = i % g_eff;
      const unsigned char* mrow = p.mask + b * p.msb + (int64_t)(s0 + ps) * p.mss;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int kk = pkt * C::BN + e * 32 + lane;
        pre_m[e] = kk < p.N ? mrow[kk * p.msk] : 0;
      }
    };
    prefetch_mask(0);
    for (int kt = 0; kt < nkt && ok; ++kt) {
      for (int s = 0; s < g_eff; ++s) {
        const int i = kt * g_eff + s;
        const int st = i % C::NS;
        if (i >= C::NS) ok = mbar_wait(&bar_kv_empty[st], ((i / C::NS) - 1) & 1, wctx);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        // additive key mask of (s, kt) in units of T (logit * sqrt(D)): 0
        // kept, -1e9*sqrt(D) masked, -inf beyond N; and a flag telling the
        // softmax whether the tile has any such key
        float* madd = reinterpret_cast<float*>(smem + C::OFF_MADD + st * C::BN * 4);
        bool any = false;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kk = kt * C::BN + e * 32 + lane;
          float a = 0.f;
          if (kk >= p.N) a = -INFINITY;
          else if (p.mask && !pre_m[e]) a = kMaskBias * sqrtf((float)D);
          madd[e * 32 + lane] = a;
          any |= a != 0.f;
        }
        any = __any_sync(0xffffffffu, any);
        if (lane == 0) *reinterpret_cast<int*>(smem + C::OFF_FLAG + st * 16) = any ? 1 : 0;
        prefetch_mask(i + 1);
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(&bar_kv_full[st], 2 * C::TILE);
        __syncwarp();
        if (lane == (rr & 31))
          tma_load_5d(smem + C::OFF_K + st * C::TILE, &tm_k, &bar_kv_full[st], 0, kt * C::BN, h,
                      s0 + s, b);
        if (lane == ((rr + 1) & 31))
          tma_load_5d(smem + C::OFF_V + st * C::TILE, &tm_v, &bar_kv_full[st], 0, kt * C::BN, h,
                      s0 + s, b);
        rr += 2;
        kv_issued = i + 1;
      }
    }
    // After a give-up, let every copy already issued land before the CTA may
    // exit (those waits end by themselves: a copy does not depend on the
    // other roles).
    if (!ok && lane == 0) {
      volatile int no_abort = 0;
      for (int i = max(0, kv_issued - C::NS); i < kv_issued; ++i)
        mbar_wait(&bar_kv_full[i % C::NS], (i / C::NS) & 1, &no_abort);
      mbar_wait(&bar_q, 0, &no_abort);
    }
    __syncwarp();
  } else if (warp == 3) {
    // =================== TMA producer of the bias tiles (one lane) =========
    // Its own warp, so that the K/V stream never waits for a bias stage.  A
    // stage is free once the MMAs of every row of kt - 2 have read it.
    if (lane == 0) {
      bool ok = true;
      int issued = 0;
      for (int kt = 0; kt < nkt && ok; ++kt) {
        const int bs = kt & 1;
        if (kt >= 2) ok = mbar_wait(&bar_bias_empty[bs], ((kt >> 1) - 1) & 1, wctx);
        if (!ok) break;
        uint8_t* dst = smem + C::OFF_BIAS + bs * C::BIAS_TILE;
        mbar_arrive_expect_tx(&bar_bias_full[bs], C::BIAS_TILE);
        if (BIAS_K_CONTIG) {  // rows j, keys contiguous
          tma_load_4d(dst, &tm_bias, &bar_bias_full[bs], kt * C::BN, jt * C::BM, h, b);
          tma_load_4d(dst + C::BIAS_TILE / 2, &tm_bias, &bar_bias_full[bs], kt * C::BN + 64,
                      jt * C::BM, h, b);
        } else {              // rows k, queries contiguous
          tma_load_4d(dst, &tm_bias, &bar_bias_full[bs], jt * C::BM, kt * C::BN, h, b);
          tma_load_4d(dst + C::BIAS_TILE / 2, &tm_bias, &bar_bias_full[bs], jt * C::BM + 64,
                      kt * C::BN, h, b);
        }
        issued = kt + 1;
      }
      if (!ok) {  // let the copies already issued land
        volatile int no_abort = 0;
        for (int kt = max(0, issued - 2); kt < issued; ++kt)
          mbar_wait(&bar_bias_full[kt & 1], (kt >> 1) & 1, &no_abort);
      }
    }
    __syncwarp();
  } else if (warp <= 2) {
    // =================== MMA issuers ======================================
    // Warp 1 issues T of every tile, warp 2 O += P V of every tile, both in
    // tile order i = kt*g_eff + s (row s belongs to softmax warpgroup s & 1).
    // Each waits (suspended in mbarrier.try_wait) for exactly the events its
    // next MMAs need, so a T waits only for its K/V stage, its bias tile and
    // the PV that frees its buffer, and a PV only for its P.  The whole warp
    // runs the loop (descriptors stay warp-uniform); the elected lane, the
    // same one throughout (the warp stays converged), issues each
    // tcgen05.mma and commit.
    const uint64_t dk0 = umma_desc(smem_u32(smem + C::OFF_K), 16, C::ATOM, C::SW);
    const uint64_t dv0 = umma_desc(smem_u32(smem + C::OFF_V), 16, C::ATOM, C::SW);
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bar_q, 0, wctx));
    if (warp == 1) {
      constexpr uint32_t id_s = idesc_bf16(128, 128, 0, 0);  // Q, K both K-major
      constexpr uint32_t id_b = idesc_bf16(128, 128, 0, BIAS_K_CONTIG ? 1 : 0);
      const uint64_t dq0 = umma_desc(smem_u32(smem + C::OFF_Q), 16, C::ATOM, C::SW);
      const uint64_t dz0 = umma_desc(smem_u32(smem + C::OFF_Z), 16, 256, kSw32);
      // bias tile as the B operand (N = keys, K = queries j'): keys contiguous
      // -> MN-major, 64-key halves 16 KB apart, 8 j'-rows per 1 KB; queries
      // contiguous -> K-major rows of 64 j' per 128 B, halves 16 KB apart
      const uint64_t dbias0 = BIAS_K_CONTIG
                                  ? umma_desc(smem_u32(smem + C::OFF_BIAS), 16384, 1024, kSw128)
                                  : umma_desc(smem_u32(smem + C::OFF_BIAS), 16, 1024, kSw128);
      for (int kt = 0, i = 0; kt < nkt && ok; ++kt) {
        for (int s = 0; s < g_eff; ++s, ++i) {
          const int st = i % C::NS, buf = i % C::NT;
          ok = mbar_wait(&bar_kv_full[st], (i / C::NS) & 1, wctx);
          if (ok && i >= C::NT) ok = mbar_wait(&bar_s_free[buf], ((i / C::NT) - 1) & 1, wctx);
          if (ok && s == 0) ok = mbar_wait(&bar_bias_full[kt & 1], (kt >> 1) & 1, wctx);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          const uint32_t tb = tmem + 128 * buf;
          const uint64_t dq = dq0 + ((uint32_t)(s * C::TILE) >> 4);
          const uint64_t dk = dk0 + ((uint32_t)(st * C::TILE) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            if (elect_one()) umma_ss(tb, dq + 2 * kk, dk + 2 * kk, id_s, kk > 0);
          const uint64_t db = dbias0 + ((uint32_t)((kt & 1) * C::BIAS_TILE) >> 4);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t a = dz0 + ((uint32_t)((112 - 16 * kk) * 32) >> 4);
            const uint64_t bb = BIAS_K_CONTIG
                                    ? db + ((uint32_t)(kk * 2048) >> 4)
                                    : db + ((uint32_t)((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
            if (elect_one()) umma_ss(tb, a, bb, id_b, 1u);
          }
          if (elect_one()) {
            umma_commit(&bar_s_full[buf]);
            if (s == g_eff - 1) umma_commit(&bar_bias_empty[kt & 1]);
          }
          __syncwarp();
        }
      }
    } else {
      constexpr uint32_t id_o = idesc_bf16(128, D, 0, 1);  // P from TMEM, V MN-major
      for (int kt = 0, i = 0; kt < nkt && ok; ++kt) {
        for (int s = 0; s < g_eff; ++s, ++i) {
          const int buf = i % C::NT;
          ok = __all_sync(0xffffffffu, mbar_wait(&bar_p_ready[buf], (i / C::NT) & 1, wctx));
          if (!ok) break;
          tc_fence_after();
          const int st = i % C::NS;
          const uint64_t dv = dv0 + ((uint32_t)(st * C::TILE) >> 4);
          const uint32_t o = tmem + C::TMEM_O + s * D, pa = tmem + 128 * buf;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            if (elect_one())
              umma_ts(o, pa + kk * 8, dv + kk * (16 * C::ROW >> 4), id_o,
                      (kt > 0 || kk > 0) ? 1u : 0u);
          if (elect_one()) {
            umma_commit(&bar_kv_empty[st]);
            umma_commit(&bar_o_done[s]);
            umma_commit(&bar_s_free[buf]);
          }
          __syncwarp();
        }
      }
    }
    // every issued MMA completes before TMEM can be released
    if (elect_one()) umma_commit(&bar_drain[warp - 1]);
    __syncwarp();
    if (lane == 0) {
      volatile int no_abort = 0;
      mbar_wait(&bar_drain[warp - 1], 0, &no_abort);
    }
    __syncwarp();
  }
  teardown();
  } else {
    // =================== softmax warpgroups ================================
    regs_inc<C::REGS_HIGH>();
    const int wg = (warp - 4) >> 2;                  // 0 or 1
    const int quad = warp & 3;                       // TMEM lane quadrant
    const int row = quad * 32 + lane;                // query row within the tile
    const int j = jt * C::BM + row;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    const float c1 = kLog2e / sqrtf((float)D);       // T to log2 units
    const float2 c1c1 = make_float2(c1, c1);
    const float lazy_thr = 8.0f / c1;                // 2^8 in probability, in T units
    float m_run[C::G / 2], l_run[C::G / 2];          // running max (T units) and sum
#pragma unroll
    for (int u = 0; u < C::G / 2; ++u) { m_run[u] = -INFINITY; l_run[u] = 0.f; }
    bool ok = wg < n_wg;
    if (ok && p.wc.stall) ok = __all_sync(0xffffffffu, stall_wait(&bar_never, wctx));
    for (int kt = 0; kt < nkt && ok; ++kt) {
#pragma unroll
      for (int u = 0; u < C::G / 2; ++u) {
        const int s = 2 * u + wg;
        if (s >= g_eff) break;
        const int i = kt * g_eff + s;
        const int st = i % C::NS;
        const uint32_t tcol = lane_base + 128 * (i % C::NT);  // T of this tile, then P
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_s_full[i % C::NT], (i / C::NT) & 1, wctx));
        if (!ok) break;
        tc_fence_after();
        uint32_t x[128];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(tcol + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&x[32 * c]));
        tmem_wait_ld();
        // key mask (warp-uniform flag: most tiles have no masked key), then
        // the row max over 4 independent chains
        if (*reinterpret_cast<const int*>(smem + C::OFF_FLAG + st * 16) != 0) {
          const float* madd = reinterpret_cast<const float*>(smem + C::OFF_MADD + st * C::BN * 4);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float4 m4 = *reinterpret_cast<const float4*>(madd + 4 * c);
            const float2 a = add2(make_float2(__uint_as_float(x[4 * c]), __uint_as_float(x[4 * c + 1])),
                                  make_float2(m4.x, m4.y));
            const float2 bq = add2(make_float2(__uint_as_float(x[4 * c + 2]), __uint_as_float(x[4 * c + 3])),
                                   make_float2(m4.z, m4.w));
            x[4 * c] = __float_as_uint(a.x); x[4 * c + 1] = __float_as_uint(a.y);
            x[4 * c + 2] = __float_as_uint(bq.x); x[4 * c + 3] = __float_as_uint(bq.y);
          }
        }
        float mx[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) mx[e] = -INFINITY;
#pragma unroll
        for (int k2 = 0; k2 < 128; k2 += 2)
          mx[(k2 >> 1) & 3] = fmax3(mx[(k2 >> 1) & 3], __uint_as_float(x[k2]), __uint_as_float(x[k2 + 1]));
        const float rmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        // The reference max m moves only when the tile's max exceeds it by
        // more than 2^8 in probability: P then stays <= 256, exact in fp32
        // and at full relative precision in bf16, and most tiles skip the O
        // rescale.  Any m gives the same softmax.
        const float m_new = rmax > m_run[u] + lazy_thr ? rmax : m_run[u];
        const float alpha = ex2((m_run[u] - m_new) * c1);
        // rescale O of this row when its running max moved (warp-uniform)
        if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bar_o_done[s], (kt - 1) & 1, wctx));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            uint32_t o[16];
            tmem_ld16(lane_base + C::TMEM_O + s * D + 16 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st16(lane_base + C::TMEM_O + s * D + 16 * c, o);
          }
        }
        // P = exp2(c1 (T - m)) as bf16 pairs over the first 64 columns of the
        // tile's T buffer (all of T is in registers by now)
        const float2 negm = make_float2(-m_new * c1, -m_new * c1);
        float2 sum[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) sum[e] = make_float2(0.f, 0.f);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int k2 = 32 * q4 + 2 * e;
            const float2 a = fma2(make_float2(__uint_as_float(x[k2]), __uint_as_float(x[k2 + 1])),
                                  c1c1, negm);
            const float2 pr = make_float2(ex2(a.x), ex2(a.y));
            sum[e & 3] = add2(sum[e & 3], pr);
            pk[e] = pack_bf16(pr.x, pr.y);
          }
          tmem_st16(tcol + 16 * q4, pk);
        }
        const float2 s01 = add2(sum[0], sum[1]), s23 = add2(sum[2], sum[3]);
        l_run[u] = l_run[u] * alpha + ((s01.x + s01.y) + (s23.x + s23.y));
        m_run[u] = m_new;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bar_p_ready[i % C::NT]);
      }
    }
    // ---- epilogue: O / l, sigmoid gate, lse -------------------------------
    // the gate rows of every row s of this warpgroup are requested before
    // the first wait, so their latency overlaps the last PV products
    uint4 gq[C::G / 2][D / 8];
    if (HAS_GATE && ok && j < p.N) {
#pragma unroll
      for (int u = 0; u < C::G / 2; ++u) {
        const int s = 2 * u + wg;
        if (s >= g_eff) break;
        const __nv_bfloat16* gsrc = p.gate + p.g.at(b, s0 + s, h, j, 0);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) gq[u][c] = *reinterpret_cast<const uint4*>(gsrc + 8 * c);
      }
    }
    if (ok) {
#pragma unroll
      for (int u = 0; u < C::G / 2; ++u) {
        const int s = 2 * u + wg;
        if (s >= g_eff) break;
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_o_done[s], (nkt - 1) & 1, wctx));
        if (!ok) break;
        tc_fence_after();
        float o[D];
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          uint32_t r[16];
          tmem_ld16(lane_base + C::TMEM_O + s * D + 16 * c, r);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) o[16 * c + e] = __uint_as_float(r[e]);
        }
        if (j < p.N) {
          const float inv_l = 1.0f / l_run[u];
          const int ss = s0 + s;
          const int64_t row_id = (((int64_t)b * p.S + ss) * p.H + h) * p.N + j;
          p.lse[row_id] = (m_run[u] * c1 + __log2f(l_run[u])) * kLn2;
          __nv_bfloat16* dst = p.out + p.o.at(b, ss, h, j, 0);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) {
            float gv[8];
            if (HAS_GATE) {
              const uint4 g4 = gq[u][c];
              gv[0] = bf16lo(g4.x); gv[1] = bf16hi(g4.x); gv[2] = bf16lo(g4.y); gv[3] = bf16hi(g4.y);
              gv[4] = bf16lo(g4.z); gv[5] = bf16hi(g4.z); gv[6] = bf16lo(g4.w); gv[7] = bf16hi(g4.w);
#pragma unroll
              for (int e = 0; e < 8; ++e) gv[e] = __fdividef(inv_l, 1.0f + ex2(-gv[e] * kLog2e));
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) gv[e] = inv_l;
            }
            uint4 w4;
            w4.x = pack_bf16(o[8 * c + 0] * gv[0], o[8 * c + 1] * gv[1]);
            w4.y = pack_bf16(o[8 * c + 2] * gv[2], o[8 * c + 3] * gv[3]);
            w4.z = pack_bf16(o[8 * c + 4] * gv[4], o[8 * c + 5] * gv[5]);
            w4.w = pack_bf16(o[8 * c + 6] * gv[6], o[8 * c + 7] * gv[7]);
            *reinterpret_cast<uint4*>(dst + 8 * c) = w4;
          }
        }
      }
    }
    teardown();
  }
}

// 5-D tensor map of a [B,S,H,N,D] bf16 view, box = 128 rows x D.
bool tmap_rows(CUtensorMap* m, const void* base, const Strides5& st, const Problem& P) {
  const uint64_t dims[5] = {(uint64_t)P.D, (uint64_t)P.N, (uint64_t)P.H, (uint64_t)P.S,
                            (uint64_t)P.B};
  const uint64_t str[4] = {(uint64_t)st.n * 2, (uint64_t)st.h * 2, (uint64_t)st.s * 2,
                           (uint64_t)st.b * 2};
  const uint32_t box[5] = {(uint32_t)P.D, 128, 1, 1, 1};
  const CUtensorMapSwizzle sw = P.D == 16 ? CU_TENSOR_MAP_SWIZZLE_32B
                                : P.D == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                            : CU_TENSOR_MAP_SWIZZLE_128B;
  return make_tmap_bf16(m, base, 5, dims, str, box, sw);
}

// 4-D tensor map of the pair bias with its contiguous axis innermost; box =
// 64 (contiguous axis) x 128, 128-byte swizzle.
bool tmap_bias(CUtensorMap* m, const void* base, const StridesBias& sb, const Problem& P,
               bool k_contig) {
  const uint64_t dims[4] = {(uint64_t)P.N, (uint64_t)P.N, (uint64_t)P.H, (uint64_t)P.B};
  const uint64_t outer = k_contig ? sb.j : sb.k;
  const uint64_t str[3] = {outer * 2, (uint64_t)sb.h * 2, (uint64_t)sb.b * 2};
  const uint32_t box[4] = {64, 128, 1, 1};
  return make_tmap_bf16(m, base, 4, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int D, bool KC, bool GATE>
cudaError_t launch_fwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const CUtensorMap& bias, const FwdParams& fp, unsigned grid,
                       cudaStream_t st) {
  using C = FwdCfg<D>;
  auto kern = evoattn_fwd_kernel<D, KC, GATE>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  // The warpgroups' register split must fit the pool the CTA is launched
  // with, or the raising warpgroups would wait forever.
  cudaFuncAttributes fa{};
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs < C::LAUNCH_REGS) return cudaErrorInvalidConfiguration;
  kern<<<grid, C::THREADS, C::SMEM_ALLOC, st>>>(q, k, v, bias, fp);
  return cudaGetLastError();
}

template <int D>
cudaError_t fwd_d(const Problem& P, const Bf16Ptrs& a, const WaitCfg& wait, cudaStream_t st,
                  bool* tmap_ok) {
  using C = FwdCfg<D>;
  CUtensorMap tq, tk, tv, tb;
  const bool kc = P.bias.k == 1;
  if (!tmap_rows(&tq, a.q, P.q, P) || !tmap_rows(&tk, a.k, P.k, P) ||
      !tmap_rows(&tv, a.v, P.v, P) || !tmap_bias(&tb, a.bias, P.bias, P, kc)) {
    *tmap_ok = false;
    return cudaErrorInvalidValue;
  }
  FwdParams fp{};
  fp.B = P.B; fp.S = P.S; fp.H = P.H; fp.N = P.N;
  fp.n_jt = (P.N + C::BM - 1) / C::BM;
  fp.n_kt = (P.N + C::BN - 1) / C::BN;
  fp.n_sg = (P.S + C::G - 1) / C::G;
  fp.mask = a.mask;
  fp.msb = P.mask.b; fp.mss = P.mask.s; fp.msk = P.mask.k;
  fp.gate = static_cast<const __nv_bfloat16*>(a.gate);
  fp.g = P.g;
  fp.out = static_cast<__nv_bfloat16*>(a.out);
  fp.o = P.o;
  fp.lse = a.lse;
  fp.wc = launch_wait(wait);
  const uint64_t grid64 = (uint64_t)fp.n_jt * P.H * fp.n_sg * P.B;
  if (grid64 > 0x7FFFFFFFull) return cudaErrorInvalidConfiguration;
  const unsigned grid = (unsigned)grid64;
  const bool gate = a.gate != nullptr;
  if (kc) return gate ? launch_fwd<D, true, true>(tq, tk, tv, tb, fp, grid, st)
                      : launch_fwd<D, true, false>(tq, tk, tv, tb, fp, grid, st);
  return gate ? launch_fwd<D, false, true>(tq, tk, tv, tb, fp, grid, st)
              : launch_fwd<D, false, false>(tq, tk, tv, tb, fp, grid, st);
}

}  // namespace

cudaError_t bf16_fwd(const Problem& P, const Bf16Ptrs& a, const WaitCfg& wait,
                     cudaStream_t st, bool* tmap_ok) {
  switch (P.D) {
    case 16: return fwd_d<16>(P, a, wait, st, tmap_ok);
    case 32: return fwd_d<32>(P, a, wait, st, tmap_ok);
    case 64: return fwd_d<64>(P, a, wait, st, tmap_ok);
  }
  return cudaErrorInvalidValue;
}

}  // namespace evo
