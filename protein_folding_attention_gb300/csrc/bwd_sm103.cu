// EvoAttention backward on sm_103a.
//
// MegaFold technical summary, "Methodik" section 1 "EvoFlash-3D": the
// backward pass recomputes the logits tile by tile in on-chip memory, as the
// forward does, so the B*S*H*N*N attention map never reaches HBM; its
// pair-bias term receives the gradient summed over the S rows that share it.
//
// With P = exp(x - lse), dOa = dout * sigmoid(g) and delta = rowsum(dOa * O):
//   dP = dOa V^T,  dS = P * (dP - delta),
//   dV = P^T dOa,  dK = dS^T Q / sqrt(D),  dQ = dS K / sqrt(D),
//   dbias[b,h,j,k] = sum_s dS[b,s,h,j,k],  dgate = dout * out * (1 - sigmoid(g)).
// The three reductions run along three different axes (dK, dV over query
// tiles, dQ over key tiles, dbias over s), so they are split over kernels:
//
//   k_pre    delta, dgate and dOa (bf16) per row; zeroes the fp32 dQ buffer
//   k_dkdv   CTA = (b, s, h, key tile): loops over query tiles with dK, dV
//            accumulating in tensor memory; dQ partial sums are added into
//            the fp32 buffer with vector atomics (deterministic dQ: each key
//            tile stores its partial into a slice of its own instead)
//   k_dbias  CTA = (b, h, query tile, key tile, s-slot): loops over the s of
//            its slot, recomputing S and dP, accumulating dS in tensor memory;
//            writes one partial per slot (or adds it atomically)
//   k_reduce ordered sum of the slot partials -> dbias; fp32 dQ (the slices
//            summed in key-tile order) -> bf16 dq
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "layout.cuh"
#include "sm103.h"
#include "tmap.h"

namespace evo {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// No memory clobber: the kernels that reduce into a buffer never read it
// back (a later kernel does), so the compiler may move other memory accesses
// across these (measured ~0.6 % on k_dkdv).
__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d));
}

// ---------------------------------------------------------------------------
// Workspace layout
// ---------------------------------------------------------------------------
inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Number of s-slots of the dbias reduction: enough CTAs for a few waves on a
// 152-SM part, fixed by the problem shape alone (so the summation order, and
// hence every bit of dbias, does not depend on the device).
inline int dbias_slots(const Problem& P) {
  const int nt = (P.N + 127) / 128;
  const long tiles = (long)P.B * P.H * nt * nt;
  long slots = (4L * 152 + tiles - 1) / tiles;
  if (slots < 1) slots = 1;
  if (slots > P.S) slots = P.S;
  return (int)slots;
}

struct Workspace {
  __nv_bfloat16* dOa;  // [B,S,H,N,D], dense in the memory order of out
  float* delta;        // [B,S,H,N]
  float* dq_acc;       // [dq_slices, B,S,H,N,D] dense fp32
  int dq_slices;       // 1 (atomic sums) or one per key tile (deterministic dQ)
  float* partial;      // [slots, B, H, N, N] fp32 (deterministic mode)
  size_t bytes;
};

Workspace carve(const Problem& P, unsigned flags, void* base) {
  const size_t L = (size_t)P.rows() * P.D;
  size_t off = 0;
  Workspace w{};
  uint8_t* b = static_cast<uint8_t*>(base);
  w.dOa = reinterpret_cast<__nv_bfloat16*>(b + off); off = align256(off + L * 2);
  w.delta = reinterpret_cast<float*>(b + off); off = align256(off + (size_t)P.rows() * 4);
  w.dq_slices = (flags & EVOATTN_DQ_DETERMINISTIC) ? (P.N + 127) / 128 : 1;
  w.dq_acc = reinterpret_cast<float*>(b + off);
  off = align256(off + (size_t)w.dq_slices * L * 4);
  w.partial = reinterpret_cast<float*>(b + off);
  if (!(flags & (EVOATTN_DBIAS_ATOMIC | EVOATTN_DBIAS_FUSED)))
    off = align256(off + (size_t)dbias_slots(P) * P.B * P.H * P.N * P.N * 4);
  w.bytes = off;
  return w;
}

// ---------------------------------------------------------------------------
// k_pre: per row, D/8 threads of 8 features each.  Rows are walked in the
// memory order of out (its s, h, n strides sorted), so that the loads of
// out, dout and the gate and the stores of dgate and dOa (laid out the same
// way) are contiguous runs whatever view the caller passes; the ending-node
// view, with n the outermost storage axis, would otherwise make every row a
// separate 64-byte access.
// ---------------------------------------------------------------------------
struct PreParams {
  int B, S, H, N, D;
  const __nv_bfloat16 *out, *dout, *gate;
  Strides5 o, dO, g, dg, a;  // a: dOa
  int walk_dim[3];           // axes (0 = s, 1 = h, 2 = n), fastest first
  int walk_size[3];
  __nv_bfloat16* dgate;
  __nv_bfloat16* dOa;
  float* delta;
  float* dq_acc;
};

// Strides of a dense [B,S,H,N,D] array whose s, h, n axes are stored in the
// order of the given view's strides (ties keep s, h, n order), and that
// order, fastest axis first.
Strides5 dense_like(const Problem& P, const Strides5& v, int (&dim)[3], int (&size)[3]) {
  const int64_t vs[3] = {v.s, v.h, v.n};
  const int sz[3] = {P.S, P.H, P.N};
  int ord[3] = {0, 1, 2};
  for (int i = 0; i < 3; ++i)  // stable insertion sort, largest stride first
    for (int k = i; k > 0 && vs[ord[k]] > vs[ord[k - 1]]; --k) {
      const int t = ord[k]; ord[k] = ord[k - 1]; ord[k - 1] = t;
    }
  int64_t st[3];
  int64_t run = P.D;
  for (int k = 2; k >= 0; --k) {  // innermost (smallest stride) first
    st[ord[k]] = run;
    run *= sz[ord[k]];
    dim[2 - k] = ord[k];
    size[2 - k] = sz[ord[k]];
  }
  return Strides5{run, st[0], st[1], st[2], 1};
}

__device__ __forceinline__ void unpack8(uint4 u, float (&f)[8]) {
  f[0] = bf16lo(u.x); f[1] = bf16hi(u.x); f[2] = bf16lo(u.y); f[3] = bf16hi(u.y);
  f[4] = bf16lo(u.z); f[5] = bf16hi(u.z); f[6] = bf16lo(u.w); f[7] = bf16hi(u.w);
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                    pack_bf16(f[6], f[7]));
}

// Each thread takes U units (row, 8 features) a grid apart and issues the
// loads of all of them before the arithmetic, so more bytes are in flight.
template <int D, int U>
__global__ void __launch_bounds__(256) k_pre(const PreParams p) {
  constexpr int TPR = D / 8;  // threads per row
  const int64_t T = (int64_t)gridDim.x * blockDim.x;  // a multiple of TPR
  const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t units = (int64_t)p.B * p.S * p.H * p.N * TPR;
  const int part = (int)(t0 % TPR);
  uint4 ro[U], rd[U], rg[U];
  int bb[U], ss[U], hh[U], jj[U];
#pragma unroll
  for (int k = 0; k < U; ++k) {
    const int64_t u = t0 + k * T;
    if (u < units) {
      const int64_t r = u / TPR;  // row in walk order
      const int i0 = (int)(r % p.walk_size[0]);
      int64_t q = r / p.walk_size[0];
      const int i1 = (int)(q % p.walk_size[1]);
      q /= p.walk_size[1];
      const int i2 = (int)(q % p.walk_size[2]);
      bb[k] = (int)(q / p.walk_size[2]);
      // axis a sits at walk position k where walk_dim[k] == a
      auto pick = [&](int a) {
        return p.walk_dim[0] == a ? i0 : (p.walk_dim[1] == a ? i1 : i2);
      };
      ss[k] = pick(0); hh[k] = pick(1); jj[k] = pick(2);
      ro[k] = *reinterpret_cast<const uint4*>(p.out + p.o.at(bb[k], ss[k], hh[k], jj[k], 8 * part));
      rd[k] = *reinterpret_cast<const uint4*>(p.dout + p.dO.at(bb[k], ss[k], hh[k], jj[k], 8 * part));
      if (p.gate)
        rg[k] = *reinterpret_cast<const uint4*>(p.gate + p.g.at(bb[k], ss[k], hh[k], jj[k], 8 * part));
    }
  }
#pragma unroll
  for (int k = 0; k < U; ++k) {
    const int64_t u = t0 + k * T;
    const bool live = u < units;
    float dl = 0.f;
    if (live) {
      const int b = bb[k], s = ss[k], h = hh[k], j = jj[k];
      float o[8], go[8], sg[8];
      unpack8(ro[k], o);
      unpack8(rd[k], go);
      if (p.gate) {
        float g[8], dg[8];
        unpack8(rg[k], g);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          sg[e] = 1.0f / (1.0f + ex2(-g[e] * kLog2e));
          dg[e] = go[e] * o[e] * (1.0f - sg[e]);
        }
        *reinterpret_cast<uint4*>(p.dgate + p.dg.at(b, s, h, j, 8 * part)) = pack8(dg);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) sg[e] = 1.0f;
      }
      float a[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        dl = fmaf(go[e], o[e], dl);
        a[e] = go[e] * sg[e];
      }
      *reinterpret_cast<uint4*>(p.dOa + p.a.at(b, s, h, j, 8 * part)) = pack8(a);
      // the fp32 dQ buffer (dense) is zeroed in unit order: 32 contiguous
      // bytes per unit (not needed when every key tile stores its own slice)
      if (p.dq_acc) {
        float4* z = reinterpret_cast<float4*>(p.dq_acc + 8 * u);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) dl += __shfl_xor_sync(0xffffffffu, dl, off);
    if (live && part == 0)
      p.delta[(((int64_t)bb[k] * p.S + ss[k]) * p.H + hh[k]) * p.N + jj[k]] = dl;
  }
}

// ---------------------------------------------------------------------------
// Shared tile configuration of the tcgen05 kernels
// ---------------------------------------------------------------------------
template <int D>
struct Tile {
  static constexpr uint32_t ROW = D * 2;
  static constexpr uint32_t ATOM = 8 * ROW;
  static constexpr Swizzle SW = D == 16 ? kSw32 : kSw64;
  static constexpr uint32_t TILE = 128 * ROW;
  static constexpr uint32_t BIAS_TILE = 128 * 128 * 2;
};

// The pair bias enters the logit tiles through the tensor core, as in the
// forward: T = Q K^T + (c I) * bias with c = sqrt(D) rounded to bf16, the
// identity never stored whole but as 128-row windows (start row 112 - 16 kk
// for reduction chunk kk) of a 240 x 16 matrix Z with Z[112 + i][i] = c,
// kept in the 32-byte-swizzled K-major layout.  The backward so recomputes
// exactly the logits whose logsumexp the forward stored.
constexpr uint32_t kZBytes = 240 * 32;
__device__ __forceinline__ void write_identity_windows(uint8_t* z, int D, int tid, int nthreads) {
  const uint32_t cb = __bfloat16_as_ushort(__float2bfloat16_rn(sqrtf((float)D)));
  uint32_t* z32 = reinterpret_cast<uint32_t*>(z);
  for (int i = tid; i < (int)(kZBytes / 4); i += nthreads) {
    const int r = i >> 3, wd = i & 7;
    const int c0 = (((wd >> 2) ^ ((r >> 2) & 1)) << 3) + ((wd & 3) << 1);
    const int one = r - 112;  // column of this row's nonzero, if any
    z32[i] = one == c0 ? cb : (one == c0 + 1 ? cb << 16 : 0u);
  }
  fence_proxy_async_smem();  // generic writes, read by the tensor core
}

// ---------------------------------------------------------------------------
// k_dkdv
// ---------------------------------------------------------------------------
// Persistent: one CTA per SM; work item = (b, s, h, key tile kt), items
// blockIdx.x, blockIdx.x + gridDim.x, ...; each item loops over the query
// tiles jt.  A global tile counter g runs across items so every ring and
// barrier phase continues from one item to the next and the producer runs
// ahead into the next item (K/V are double-buffered per item).
//
// Warps (384 threads): 0 TMA producer, 1-3 MMA issuers (S/dP, dV/dK, dQ),
// 4-11 two compute warpgroups.  A compute thread owns key k (TMEM lane 32*(warp%4)+lane) and,
// of each 128-query tile, the 64 queries of its warpgroup's half.  Tensor
// memory columns: S^T 0..127, dP^T 128..255 (fp32, lane = key), P^T 256..,
// dS^T 320.. (bf16 pairs, 32 columns per half), two dQ partial buffers
// 384.. (lane = query), dK and dV after them (lane = key).
//
template <int D, bool BIAS_K_CONTIG>
struct DkdvCfg : Tile<D> {
  using T = Tile<D>;
  static constexpr int NQ = 3;  // Q/dO/(lse,delta) stages
  static constexpr int NB = 3;  // bias stages (as the TMA delivers them)
  static constexpr uint32_t OFF_K = 0;                              // 2 stages
  static constexpr uint32_t OFF_V = OFF_K + 2 * T::TILE;            // 2 stages
  static constexpr uint32_t OFF_Q = OFF_V + 2 * T::TILE;
  static constexpr uint32_t OFF_DO = OFF_Q + NQ * T::TILE;
  static constexpr uint32_t OFF_BIAS = OFF_DO + NQ * T::TILE;
  static constexpr uint32_t OFF_DS = OFF_BIAS + NB * T::BIAS_TILE;
  static constexpr uint32_t OFF_Z = OFF_DS + 128 * 128 * 2;
  static constexpr uint32_t OFF_LD = OFF_Z + kZBytes;  // -lse2[128], -delta/sqrt(D)[128]
  static constexpr uint32_t SMEM = OFF_LD + NQ * 256 * 4;
  static constexpr uint32_t SMEM_ALLOC = SMEM + 1024;
  static constexpr uint32_t T_S = 0, T_DP = 128, T_P = 256, T_DS = 320, T_DQ = 384,
                            T_DK = 384 + 2 * D, T_DV = 384 + 3 * D;
  static_assert(T_DV + D <= 512, "tensor memory overflow");
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory overflow");
  static_assert(OFF_BIAS % 1024 == 0 && OFF_DS % 1024 == 0 && OFF_Z % 256 == 0, "alignment");
  static constexpr int THREADS = 384;
  static constexpr int LAUNCH_REGS = 168, REGS_LOW = 56, REGS_HIGH = 216;
  static_assert(REGS_LOW * 128 + REGS_HIGH * 256 <= LAUNCH_REGS * THREADS, "register split");
};

struct DkdvParams {
  int B, S, H, N, njt, nkt, n_items;
  const unsigned char* mask;
  int64_t msb, mss, msk;
  const float* lse;
  const float* delta;
  float* dq_acc;
  // deterministic dQ: key tile kt stores its partial, plain, into slice kt
  // (slice stride dq_slice elements) instead of adding it atomically
  int dq_det;
  int64_t dq_slice;
  __nv_bfloat16 *dk, *dv;
  Strides5 sdk, sdv;
  float* dbias;  // fused dbias: dense fp32 [B,H,N,N], zeroed before the launch
  WaitCfg wc;
};

struct DkdvItem {
  int b, s, h, kt;
  int64_t row0;  // row of (b, s, h, 0) in a dense [B,S,H,N] array
};

// FUSED_DBIAS: the logit gradients are also added into dbias (fp32 atomics)
// here, so no second pass recomputes them.
template <int D, bool BIAS_K_CONTIG, bool FUSED_DBIAS>
__global__ void __launch_bounds__(384, 1)
    k_dkdv(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
           const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
           const __grid_constant__ CUtensorMap tm_bias, const DkdvParams p) {
  using C = DkdvCfg<D, BIAS_K_CONTIG>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bar_kv_full[2], bar_kv_empty[2], bar_qd_full[C::NQ], bar_qd_empty[C::NQ],
      bar_b_full[C::NB], bar_b_empty[C::NB], bar_s_full, bar_sdp_free, bar_p_ready,
      bar_mma_done, bar_dq_free[2], bar_dkdv_free, bar_drain[3], bar_never;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int njt = p.njt;
  const int my_items = (p.n_items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  const int total = my_items * njt;  // tiles of this CTA
  auto item = [&](int n) -> DkdvItem {
    int idx = (int)blockIdx.x + n * (int)gridDim.x;
    DkdvItem it;
    it.kt = idx % p.nkt; idx /= p.nkt;
    it.h = idx % p.H; idx /= p.H;
    it.s = idx % p.S;
    it.b = idx / p.S;
    it.row0 = (((int64_t)it.b * p.S + it.s) * p.H + it.h) * p.N;
    return it;
  };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_kv_full[i], 1); mbar_init(&bar_kv_empty[i], 1);
      // one "read" barrier per dQ buffer: a single barrier could complete two
      // phases (tiles g-2 and g-1) before the MMA thread looks at it
      mbar_init(&bar_dq_free[i], 256);
    }
    for (int i = 0; i < C::NQ; ++i) { mbar_init(&bar_qd_full[i], 1); mbar_init(&bar_qd_empty[i], 1); }
    // a bias stage is free once the MMAs of its tile have read it
    for (int i = 0; i < C::NB; ++i) { mbar_init(&bar_b_full[i], 1); mbar_init(&bar_b_empty[i], 1); }
    mbar_init(&bar_s_full, 1); mbar_init(&bar_sdp_free, 256); mbar_init(&bar_p_ready, 256);
    // dV/dK and dQ of a tile are committed by two issuers
    mbar_init(&bar_mma_done, 2); mbar_init(&bar_dkdv_free, 256);
    for (int i = 0; i < 3; ++i) mbar_init(&bar_drain[i], 1);
    mbar_init(&bar_never, 1);  // nothing arrives: the stall test waits on it
    fence_barrier_init();
  }
  write_identity_windows(smem + C::OFF_Z, D, threadIdx.x, C::THREADS);
  if (warp == 1) tmem_alloc(&tmem_slot, 512);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q); tma_prefetch_desc(&tm_k); tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do); tma_prefetch_desc(&tm_bias);
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

  if (warp < 4) {
  // setmaxnreg is warpgroup-aligned: one instance for warps 0-3, one for 4-11
  regs_dec<C::REGS_LOW>();
  if (warp == 0) {
    // ============================ producer =================================
    // The bias tile goes to its stage as the TMA delivers it (the MMA reads
    // either layout).  Copies issued by one thread are served in order, those of different
    // threads concurrently: each box is issued by the next lane in turn (the
    // whole warp calls issue_bias; lane 0 arms the barrier first).
    int rr = 0;
    auto issue_bias = [&](int g, uint8_t* dst, uint64_t* bar) {
      const DkdvItem it = item(g / njt);
      const int jt = g % njt;
      if (lane == 0) mbar_arrive_expect_tx(bar, C::BIAS_TILE);
      __syncwarp();
      const int l0 = rr & 31, l1 = (rr + 1) & 31;
      rr += 2;
      if (BIAS_K_CONTIG) {
        if (lane == l0) tma_load_4d(dst, &tm_bias, bar, it.kt * 128, jt * 128, it.h, it.b);
        if (lane == l1) tma_load_4d(dst + 16384, &tm_bias, bar, it.kt * 128 + 64, jt * 128, it.h, it.b);
      } else {
        if (lane == l0) tma_load_4d(dst, &tm_bias, bar, jt * 128, it.kt * 128, it.h, it.b);
        if (lane == l1) tma_load_4d(dst + 16384, &tm_bias, bar, jt * 128 + 64, it.kt * 128, it.h, it.b);
      }
    };
    const float inv_sqrt_d = rsqrtf((float)D);
    bool ok = true;
    int kv_issued = 0, qd_issued = 0, b_issued = 0;
    // The per-query constants of tile g+1 are loaded into registers while
    // tile g is being armed, so the producer never waits on their latency.
    float pre_l[4], pre_d[4];
    auto prefetch = [&](int t) {
      if (t >= total) return;
      const DkdvItem pt = item(t / njt);
      const int pjt = t % njt;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = pjt * 128 + e * 32 + lane;
        pre_l[e] = j < p.N ? p.lse[pt.row0 + j] : 0.f;
        pre_d[e] = j < p.N ? p.delta[pt.row0 + j] : 0.f;
      }
    };
    prefetch(0);
    int g = 0;
    for (int n = 0; n < my_items && ok; ++n) {
      const DkdvItem it = item(n);
      const int kvs = n & 1;
      if (n >= 2) ok = mbar_wait(&bar_kv_empty[kvs], ((n >> 1) - 1) & 1, wctx);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (lane == 0) mbar_arrive_expect_tx(&bar_kv_full[kvs], 2 * C::TILE);
      __syncwarp();
      if (lane == (rr & 31))
        tma_load_5d(smem + C::OFF_K + kvs * C::TILE, &tm_k, &bar_kv_full[kvs], 0, it.kt * 128,
                    it.h, it.s, it.b);
      if (lane == ((rr + 1) & 31))
        tma_load_5d(smem + C::OFF_V + kvs * C::TILE, &tm_v, &bar_kv_full[kvs], 0, it.kt * 128,
                    it.h, it.s, it.b);
      rr += 2;
      kv_issued = n + 1;
      for (int jt = 0; jt < njt; ++jt, ++g) {
        const int qs = g % C::NQ, bs = g % C::NB;
        if (g >= C::NQ) ok = mbar_wait(&bar_qd_empty[qs], ((g / C::NQ) - 1) & 1, wctx);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        // Q and dOa tiles first; the phase completes only with the arrival
        // after the per-query constants below
        if (lane == 0) mbar_expect_tx(&bar_qd_full[qs], 2 * C::TILE);
        __syncwarp();
        if (lane == (rr & 31))
          tma_load_5d(smem + C::OFF_Q + qs * C::TILE, &tm_q, &bar_qd_full[qs], 0, jt * 128, it.h,
                      it.s, it.b);
        if (lane == ((rr + 1) & 31))
          tma_load_5d(smem + C::OFF_DO + qs * C::TILE, &tm_do, &bar_qd_full[qs], 0, jt * 128,
                      it.h, it.s, it.b);
        rr += 2;
        // per-query constants of this tile, negated: -lse in log2 units
        // (-inf beyond N so that P = 0 there) and -delta / sqrt(D)
        float* ld = reinterpret_cast<float*>(smem + C::OFF_LD + qs * 1024);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int jl = e * 32 + lane, j = jt * 128 + jl;
          ld[jl] = j < p.N ? -pre_l[e] * kLog2e : -INFINITY;
          ld[128 + jl] = j < p.N ? -pre_d[e] * inv_sqrt_d : 0.f;
        }
        prefetch(g + 1);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_qd_full[qs]);
        qd_issued = g + 1;
        if (g >= C::NB) ok = mbar_wait(&bar_b_empty[bs], ((g / C::NB) - 1) & 1, wctx);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        issue_bias(g, smem + C::OFF_BIAS + bs * C::BIAS_TILE, &bar_b_full[bs]);
        b_issued = g + 1;
      }
    }
    // After a give-up, let every copy already issued land before the CTA may
    // exit (those waits end by themselves: a copy does not depend on the
    // other roles).
    if (!ok && lane == 0) {
      volatile int no_abort = 0;
      for (int i = max(0, kv_issued - 2); i < kv_issued; ++i)
        mbar_wait(&bar_kv_full[i & 1], (i >> 1) & 1, &no_abort);
      for (int i = max(0, qd_issued - C::NQ); i < qd_issued; ++i)
        mbar_wait(&bar_qd_full[i % C::NQ], (i / C::NQ) & 1, &no_abort);
      for (int i = max(0, b_issued - C::NB); i < b_issued; ++i)
        mbar_wait(&bar_b_full[i % C::NB], (i / C::NB) & 1, &no_abort);
    }
    __syncwarp();
  } else {
    // ============================ MMA issuers ==============================
    // Warp 1 issues S^T / dP^T, warp 2 dV and dK, warp 3 dQ.  Each waits
    // (suspended in mbarrier.try_wait) for exactly what its next MMAs need,
    // so the small N = D products of one tile go out from two threads at
    // once and none of them waits behind another's dependencies.  The whole
    // warp runs the loop (descriptors stay warp-uniform); the elected lane,
    // the same one throughout, issues each tcgen05.mma and commit.
    constexpr uint32_t TILE16 = C::TILE >> 4, KSTEP16 = (16 * C::ROW) >> 4;
    bool ok = true;
    if (warp == 1) {
      // S^T = K Q^T + (c I) bias^T and dP^T = V dOa^T once Q/dOa, the bias
      // tile (and, on an item's first tile, K/V) are loaded and S/dP of the
      // previous tile are in the compute threads' registers
      constexpr uint32_t id_sdp = idesc_bf16(128, 128, 0, 0);  // A=K/V, B=Q/dOa, K-major
      // bias tile as the B operand (N = queries j, K = keys k'): keys
      // contiguous -> K-major rows of 64 k' per 128 B, halves 16 KB apart;
      // queries contiguous -> MN-major, 64-query halves 16 KB apart, 8
      // k'-rows per 1 KB
      constexpr uint32_t id_b = idesc_bf16(128, 128, 0, BIAS_K_CONTIG ? 0 : 1);
      const uint64_t dk0 = umma_desc(smem_u32(smem + C::OFF_K), 16, C::ATOM, C::SW);
      const uint64_t dv0 = umma_desc(smem_u32(smem + C::OFF_V), 16, C::ATOM, C::SW);
      const uint64_t dq0 = umma_desc(smem_u32(smem + C::OFF_Q), 16, C::ATOM, C::SW);
      const uint64_t ddo0 = umma_desc(smem_u32(smem + C::OFF_DO), 16, C::ATOM, C::SW);
      const uint64_t dz0 = umma_desc(smem_u32(smem + C::OFF_Z), 16, 256, kSw32);
      const uint64_t dbias0 = BIAS_K_CONTIG
                                  ? umma_desc(smem_u32(smem + C::OFF_BIAS), 16, 1024, kSw128)
                                  : umma_desc(smem_u32(smem + C::OFF_BIAS), 16384, 1024, kSw128);
      int g = 0;
      for (int n = 0; n < my_items && ok; ++n) {
        const int kvs = n & 1;
        for (int jt = 0; jt < njt; ++jt, ++g) {
          const int qs = g % C::NQ, bs = g % C::NB;
          ok = mbar_wait(&bar_qd_full[qs], (g / C::NQ) & 1, wctx);
          if (ok && jt == 0) ok = mbar_wait(&bar_kv_full[kvs], (n >> 1) & 1, wctx);
          if (ok && g > 0) ok = mbar_wait(&bar_sdp_free, (g - 1) & 1, wctx);
          if (ok) ok = mbar_wait(&bar_b_full[bs], (g / C::NB) & 1, wctx);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dk = dk0 + kvs * TILE16, dv = dv0 + kvs * TILE16;
          const uint64_t dq = dq0 + qs * TILE16, ddo = ddo0 + qs * TILE16;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            if (elect_one()) umma_ss(tmem + C::T_S, dk + 2 * kk, dq + 2 * kk, id_sdp, kk > 0);
            if (elect_one()) umma_ss(tmem + C::T_DP, dv + 2 * kk, ddo + 2 * kk, id_sdp, kk > 0);
          }
          const uint64_t db = dbias0 + ((uint32_t)(bs * C::BIAS_TILE) >> 4);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t a = dz0 + ((uint32_t)((112 - 16 * kk) * 32) >> 4);
            const uint64_t bb = BIAS_K_CONTIG
                                    ? db + ((uint32_t)((kk >> 2) * 16384 + (kk & 3) * 32) >> 4)
                                    : db + ((uint32_t)(kk * 2048) >> 4);
            if (elect_one()) umma_ss(tmem + C::T_S, a, bb, id_b, 1u);
          }
          if (elect_one()) {
            umma_commit(&bar_s_full);
            umma_commit(&bar_b_empty[bs]);
          }
          __syncwarp();
        }
      }
    } else if (warp == 2) {
      // dV += P^T dOa and dK += dS^T Q (K dimension = queries) once P^T and
      // dS^T are stored; on an item's first tile the previous item's dK/dV
      // must have been read out
      constexpr uint32_t id_kv = idesc_bf16(128, D, 0, 1);  // A=P^T/dS^T (TMEM), B MN-major
      const uint64_t dq0 = umma_desc(smem_u32(smem + C::OFF_Q), 16, C::ATOM, C::SW);
      const uint64_t ddo0 = umma_desc(smem_u32(smem + C::OFF_DO), 16, C::ATOM, C::SW);
      int g = 0;
      for (int n = 0; n < my_items && ok; ++n) {
        for (int jt = 0; jt < njt; ++jt, ++g) {
          const int qs = g % C::NQ;
          ok = mbar_wait(&bar_p_ready, g & 1, wctx);
          if (ok && jt == 0 && n > 0) ok = mbar_wait(&bar_dkdv_free, (n - 1) & 1, wctx);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dq = dq0 + qs * TILE16, ddo = ddo0 + qs * TILE16;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t acc = (jt > 0 || kk > 0) ? 1u : 0u;
            if (elect_one())
              umma_ts(tmem + C::T_DV, tmem + C::T_P + kk * 8, ddo + kk * KSTEP16, id_kv, acc);
            if (elect_one())
              umma_ts(tmem + C::T_DK, tmem + C::T_DS + kk * 8, dq + kk * KSTEP16, id_kv, acc);
          }
          if (elect_one()) {
            umma_commit(&bar_qd_empty[qs]);
            umma_commit(&bar_mma_done);
          }
          __syncwarp();
        }
      }
    } else {
      // dQ partial = dS K (K dimension = keys) once dS is in shared memory
      // and the compute threads have read the buffer's previous partial
      constexpr uint32_t id_q = idesc_bf16(128, D, 1, 1);  // A=dS (smem, MN-major)
      const uint64_t dk0 = umma_desc(smem_u32(smem + C::OFF_K), 16, C::ATOM, C::SW);
      const uint64_t dds0 = umma_desc(smem_u32(smem + C::OFF_DS), 16384, 1024, kSw128);
      int g = 0;
      for (int n = 0; n < my_items && ok; ++n) {
        const int kvs = n & 1;
        for (int jt = 0; jt < njt; ++jt, ++g) {
          ok = mbar_wait(&bar_p_ready, g & 1, wctx);
          if (ok && g >= 2) ok = mbar_wait(&bar_dq_free[g & 1], ((g >> 1) - 1) & 1, wctx);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dk = dk0 + kvs * TILE16;
          const uint32_t dqt = tmem + C::T_DQ + (g & 1) * D;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            if (elect_one()) umma_ss(dqt, dds0 + kk * (2048 >> 4), dk + kk * KSTEP16, id_q, kk > 0);
          if (elect_one()) {
            if (jt == njt - 1) umma_commit(&bar_kv_empty[kvs]);
            umma_commit(&bar_mma_done);
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
    // ============================ compute ==================================
    regs_inc<C::REGS_HIGH>();
    const int wg = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int kl = quad * 32 + lane;          // key within the tile (TMEM lane)
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    const float c1 = kLog2e * rsqrtf((float)D);
    const float inv_sqrt_d = rsqrtf((float)D);
    const float2 c1c1 = make_float2(c1, c1), l2l2 = make_float2(kLog2e, kLog2e),
                 isd = make_float2(inv_sqrt_d, inv_sqrt_d);
    const float sqrt_d = sqrtf((float)D);
    // dQ partial of tile t (query tile jt_t of the item at row0_t, key tile
    // kt_t): lane = query; this warpgroup adds (or, deterministic, stores)
    // half of D
    auto dq_epilogue = [&](int t, int64_t row0_t, int jt_t, int kt_t) {
      uint32_t q16[D / 2];
      if constexpr (D == 32) {
        tmem_ld16(lane_base + C::T_DQ + (t & 1) * D + 16 * wg,
                  *reinterpret_cast<uint32_t(*)[16]>(&q16[0]));
      } else {
        uint32_t tmp[16];
        tmem_ld16(lane_base + C::T_DQ + (t & 1) * D, tmp);  // D = 16: each half adds 8
#pragma unroll
        for (int e = 0; e < 8; ++e) q16[e] = tmp[8 * wg + e];
      }
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bar_dq_free[t & 1]);
      const int jg = jt_t * 128 + kl;  // this lane's query row
      if (jg < p.N) {
        float* dst = p.dq_acc + (row0_t + jg) * D + (D / 2) * wg;
        if (p.dq_det) {
          float4* d4 = reinterpret_cast<float4*>(dst + kt_t * p.dq_slice);
#pragma unroll
          for (int e = 0; e < D / 2; e += 4)
            d4[e / 4] = make_float4(__uint_as_float(q16[e]), __uint_as_float(q16[e + 1]),
                                    __uint_as_float(q16[e + 2]), __uint_as_float(q16[e + 3]));
        } else {
#pragma unroll
          for (int e = 0; e < D / 2; e += 4)
            red_add_v4(dst + e, __uint_as_float(q16[e]), __uint_as_float(q16[e + 1]),
                       __uint_as_float(q16[e + 2]), __uint_as_float(q16[e + 3]));
        }
      }
    };
    // mask byte of this thread's key in item n, loaded one item ahead so its
    // latency never sits at an item boundary
    auto mask_of = [&](int n) -> int {
      if (n >= my_items || !p.mask) return 1;
      const DkdvItem mi = item(n);
      const int mk = mi.kt * 128 + kl;
      return mk < p.N ? (int)p.mask[mi.b * p.msb + (int64_t)mi.s * p.mss + (int64_t)mk * p.msk] : 1;
    };
    int mask_next = mask_of(0);
    // End of an item: its last dQ partial, then dK (warpgroup 0) and dV
    // (warpgroup 1) of its key tile.  Run after the math of the next item's
    // first tile, by which time the item's last MMAs have completed, so the
    // compute threads never idle on them at an item boundary.
    auto item_end = [&](const DkdvItem& e, int g_last) {
      dq_epilogue(g_last, e.row0, njt - 1, e.kt);
      uint32_t r[D];
      const uint32_t col = wg == 0 ? C::T_DK : C::T_DV;
#pragma unroll
      for (int c = 0; c < D / 16; ++c)
        tmem_ld16(lane_base + col + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&r[16 * c]));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bar_dkdv_free);
      const int ek = e.kt * 128 + kl;
      if (ek < p.N) {
        __nv_bfloat16* dst = wg == 0 ? p.dk + p.sdk.at(e.b, e.s, e.h, ek, 0)
                                     : p.dv + p.sdv.at(e.b, e.s, e.h, ek, 0);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          float f[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) f[q] = __uint_as_float(r[8 * c + q]);
          *reinterpret_cast<uint4*>(dst + 8 * c) = pack8(f);
        }
      }
    };
    bool ok = true, pending = false;
    if (p.wc.stall) ok = __all_sync(0xffffffffu, stall_wait(&bar_never, wctx));
    DkdvItem prev{};
    int g = 0;
    for (int n = 0; n < my_items && ok; ++n) {
      const DkdvItem it = item(n);
      const int kg = it.kt * 128 + kl;  // key index
      float* const dbias_row =
          FUSED_DBIAS ? p.dbias + ((int64_t)it.b * p.H + it.h) * p.N * p.N : nullptr;
      // additive mask of this key, log2 units (constant over the query tiles)
      float madd = 0.f;
      if (kg >= p.N) madd = -INFINITY;
      else if (!mask_next) madd = kMaskBias * kLog2e;
      mask_next = mask_of(n + 1);
      const float2 mm = make_float2(madd, madd);
      for (int jt = 0; jt < njt; ++jt, ++g) {
        const int qs = g % C::NQ;
        ok = mbar_wait(&bar_s_full, g & 1, wctx) &&
             mbar_wait(&bar_qd_full[qs], (g / C::NQ) & 1, wctx);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        uint32_t sx[64], dpx[64];
        tmem_ld32(lane_base + C::T_S + 64 * wg, *reinterpret_cast<uint32_t(*)[32]>(&sx[0]));
        tmem_ld32(lane_base + C::T_S + 64 * wg + 32, *reinterpret_cast<uint32_t(*)[32]>(&sx[32]));
        tmem_ld32(lane_base + C::T_DP + 64 * wg, *reinterpret_cast<uint32_t(*)[32]>(&dpx[0]));
        tmem_ld32(lane_base + C::T_DP + 64 * wg + 32,
                  *reinterpret_cast<uint32_t(*)[32]>(&dpx[32]));
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bar_sdp_free);
        const float* ld = reinterpret_cast<const float*>(smem + C::OFF_LD + qs * 1024);
        uint32_t pk[32], dk2[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // 8 queries per step
          const float4 la = *reinterpret_cast<const float4*>(ld + 64 * wg + 8 * c);
          const float4 lb = *reinterpret_cast<const float4*>(ld + 64 * wg + 8 * c + 4);
          const float4 da = *reinterpret_cast<const float4*>(ld + 128 + 64 * wg + 8 * c);
          const float4 db = *reinterpret_cast<const float4*>(ld + 128 + 64 * wg + 8 * c + 4);
          const float2 nl[4] = {make_float2(la.x, la.y), make_float2(la.z, la.w),
                                make_float2(lb.x, lb.y), make_float2(lb.z, lb.w)};
          const float2 nd[4] = {make_float2(da.x, da.y), make_float2(da.z, da.w),
                                make_float2(db.x, db.y), make_float2(db.z, db.w)};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j2 = 8 * c + 2 * e;
            // S already holds the pair bias (scaled by c = bf16(sqrt(D)))
            float2 t = fma2(make_float2(__uint_as_float(sx[j2]), __uint_as_float(sx[j2 + 1])),
                            c1c1, mm);
            t = add2(t, nl[e]);
            const float2 pr = make_float2(ex2(t.x), ex2(t.y));
            const float2 gg = fma2(
                make_float2(__uint_as_float(dpx[j2]), __uint_as_float(dpx[j2 + 1])), isd, nd[e]);
            const float2 ds = mul2(pr, gg);
            pk[4 * c + e] = pack_bf16(pr.x, pr.y);
            dk2[4 * c + e] = pack_bf16(ds.x, ds.y);
            if constexpr (FUSED_DBIAS) {
              // dbias[b, h, j, k] += the logit gradient (ds carries the
              // 1/sqrt(D) of dQ and dK); a warp covers 32 consecutive keys
              const int jq = jt * 128 + 64 * wg + j2;
              if (kg < p.N) {
                float* cell = dbias_row + (int64_t)jq * p.N + kg;
                if (jq < p.N) atomicAdd(cell, ds.x * sqrt_d);
                if (jq + 1 < p.N) atomicAdd(cell + p.N, ds.y * sqrt_d);
              }
            }
          }
        }
        // the previous tile's MMAs read P^T, dS^T and the dS tile: wait for them
        if (g > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bar_mma_done, (g - 1) & 1, wctx));
          if (!ok) break;
          tc_fence_after();
        }
        if (pending) {  // the previous item's last tile is g - 1
          item_end(prev, g - 1);
          pending = false;
        }
        tmem_st32(lane_base + C::T_P + 32 * wg, pk);
        tmem_st32(lane_base + C::T_DS + 32 * wg, dk2);
        // dS into shared memory as the M-major A operand of dQ = dS K: row k,
        // queries of this half contiguous, 128-byte swizzle.
        {
          uint8_t* rowp = smem + C::OFF_DS + wg * 16384 + (kl >> 3) * 1024 + (kl & 7) * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(rowp + ((c ^ (kl & 7)) << 4)) =
                make_uint4(dk2[4 * c], dk2[4 * c + 1], dk2[4 * c + 2], dk2[4 * c + 3]);
        }
        fence_proxy_async_smem();
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bar_p_ready);
        if (jt > 0) dq_epilogue(g - 1, it.row0, jt - 1, it.kt);  // its MMAs completed (waited above)
      }
      prev = it;
      pending = true;
    }
    // the last item's end
    if (ok && pending) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_mma_done, (g - 1) & 1, wctx));
      if (ok) {
        tc_fence_after();
        item_end(prev, g - 1);
      }
    }
    teardown();
  }
}

// ---------------------------------------------------------------------------
// k_dbias
// ---------------------------------------------------------------------------
// CTA = (b, h, query tile jt, key tile kt, s-slot).  Warps (640 threads): 0
// producer, 1 MMA, 2-3 idle, 4-19 four compute warpgroups; a compute thread
// owns query j (TMEM lane) and the 32 keys of its warpgroup's quarter.  Tensor
// memory: S 0..127, dP 128..255 (fp32, lane =
// query); each compute thread keeps its 32 dbias sums in registers across
// the slot's s.  The bias tile is fetched once per CTA as the TMA delivers
// it and added into every S tile by the identity-window MMAs.
template <int D>
struct DbiasCfg : Tile<D> {
  using T = Tile<D>;
  static constexpr int NST = 4;  // (Q, dOa, K, V) stages over s
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_DO = OFF_Q + NST * T::TILE;
  static constexpr uint32_t OFF_K = OFF_DO + NST * T::TILE;
  static constexpr uint32_t OFF_V = OFF_K + NST * T::TILE;
  static constexpr uint32_t OFF_BIAS = OFF_V + NST * T::TILE;
  static constexpr uint32_t OFF_Z = OFF_BIAS + T::BIAS_TILE;
  static constexpr uint32_t OFF_MADD = OFF_Z + kZBytes;
  static constexpr uint32_t OFF_FLAG = OFF_MADD + NST * 128 * 4;  // per stage: any masked key
  static constexpr uint32_t SMEM = OFF_FLAG + NST * 16;
  static constexpr uint32_t SMEM_ALLOC = SMEM + 1024;
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory overflow");
  // S and dP double-buffered: buffer b at 256 b, so the MMAs of the next s
  // run while the compute threads work on the current one
  static constexpr uint32_t T_S = 0, T_DP = 128, T_BUF = 256;
  // Four compute warpgroups, each with 32 keys of every tile: four warps per
  // sub-partition hide the element-wise work's latencies that two could not
  static constexpr int NWG = 4;                  // compute warpgroups
  static constexpr int KPT = 128 / NWG;          // keys per compute thread
  static constexpr int CH = 16;                  // keys per tensor-memory load
  static constexpr int THREADS = 128 * (1 + NWG);
  static constexpr int LAUNCH_REGS = 96, REGS_LOW = 64, REGS_HIGH = 104;
  static_assert(REGS_LOW * 128 + REGS_HIGH * 128 * NWG <= LAUNCH_REGS * THREADS,
                "register split");
};

struct DbiasParams {
  int B, S, H, N, njt, nkt, slots;
  const unsigned char* mask;
  int64_t msb, mss, msk;
  const float* lse;
  const float* delta;
  float* out;       // partial [slots,B,H,N,N] or dbias [B,H,N,N]
  int atomic;
  WaitCfg wc;
};

template <int D, bool BIAS_K_CONTIG>
__global__ void __launch_bounds__(DbiasCfg<D>::THREADS, 1)
    k_dbias(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
            const __grid_constant__ CUtensorMap tm_bias, const DbiasParams p) {
  using C = DbiasCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bar_bias, bar_full[C::NST], bar_empty[C::NST], bar_s_full[2],
      bar_sdp_free[2], bar_drain, bar_never;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  int idx = blockIdx.x;
  const int kt = idx % p.nkt; idx /= p.nkt;
  const int jt = idx % p.njt; idx /= p.njt;
  const int slot = idx % p.slots; idx /= p.slots;
  const int h = idx % p.H;
  const int b = idx / p.H;
  // contiguous s range of this slot
  const int s_begin = (int)(((int64_t)p.S * slot) / p.slots);
  const int s_end = (int)(((int64_t)p.S * (slot + 1)) / p.slots);
  const int ns = s_end - s_begin;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_bias, 1);
    // a stage is empty once its MMAs completed (one commit) and both compute
    // warpgroups are done with its key mask (256 arrivals)
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_empty[i], 1 + 128 * C::NWG);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_s_full[i], 1);
      mbar_init(&bar_sdp_free[i], 128 * C::NWG);
    }
    mbar_init(&bar_drain, 1);
    mbar_init(&bar_never, 1);  // nothing arrives: the stall test waits on it
    fence_barrier_init();
  }
  write_identity_windows(smem + C::OFF_Z, D, threadIdx.x, C::THREADS);
  if (warp == 1) tmem_alloc(&tmem_slot, 512);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q); tma_prefetch_desc(&tm_k); tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do); tma_prefetch_desc(&tm_bias);
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

  if (warp < 4) {
  // setmaxnreg is warpgroup-aligned: one instance for warps 0-3, one for 4-11
  regs_dec<C::REGS_LOW>();
  if (warp == 0) {
    // ============================ producer =================================
    bool ok = true;
    {
      // copies issued by one thread are served in order, those of different
      // threads concurrently: each box goes out from its own lane
      uint8_t* dst = smem + C::OFF_BIAS;
      uint64_t* bar = &bar_bias;
      if (lane == 0) mbar_arrive_expect_tx(bar, C::BIAS_TILE);
      __syncwarp();
      if (BIAS_K_CONTIG) {
        if (lane == 0) tma_load_4d(dst, &tm_bias, bar, kt * 128, jt * 128, h, b);
        if (lane == 1) tma_load_4d(dst + 16384, &tm_bias, bar, kt * 128 + 64, jt * 128, h, b);
      } else {
        if (lane == 0) tma_load_4d(dst, &tm_bias, bar, jt * 128, kt * 128, h, b);
        if (lane == 1) tma_load_4d(dst + 16384, &tm_bias, bar, jt * 128 + 64, kt * 128, h, b);
      }
    }
    int issued = 0;
    // mask bytes of the next s are loaded while the current one is armed
    unsigned char pre_m[4];
    auto prefetch_mask = [&](int i) {
      if (i >= ns || !p.mask) return;
      const unsigned char* mrow = p.mask + b * p.msb + (int64_t)(s_begin + i) * p.mss;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int kk = kt * 128 + e * 32 + lane;
        pre_m[e] = kk < p.N ? mrow[kk * p.msk] : 0;
      }
    };
    prefetch_mask(0);
    for (int i = 0; i < ns; ++i) {
      const int st = i % C::NST, s = s_begin + i;
      if (i >= C::NST) ok = mbar_wait(&bar_empty[st], ((i / C::NST) - 1) & 1, wctx);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      float* madd = reinterpret_cast<float*>(smem + C::OFF_MADD + st * 512);
      bool any = false;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int kk = kt * 128 + e * 32 + lane;
        float a = 0.f;
        if (kk >= p.N) a = -INFINITY;
        else if (p.mask && !pre_m[e]) a = kMaskBias * kLog2e;
        madd[e * 32 + lane] = a;
        any |= a != 0.f;
      }
      any = __any_sync(0xffffffffu, any);
      if (lane == 0) *reinterpret_cast<int*>(smem + C::OFF_FLAG + st * 16) = any ? 1 : 0;
      prefetch_mask(i + 1);
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&bar_full[st], 4 * C::TILE);
      __syncwarp();
      {
        const int l0 = (2 + 4 * i) & 31;  // lanes 0-1 issued the bias
        if (lane == l0)
          tma_load_5d(smem + C::OFF_Q + st * C::TILE, &tm_q, &bar_full[st], 0, jt * 128, h, s, b);
        if (lane == ((l0 + 1) & 31))
          tma_load_5d(smem + C::OFF_DO + st * C::TILE, &tm_do, &bar_full[st], 0, jt * 128, h, s, b);
        if (lane == ((l0 + 2) & 31))
          tma_load_5d(smem + C::OFF_K + st * C::TILE, &tm_k, &bar_full[st], 0, kt * 128, h, s, b);
        if (lane == ((l0 + 3) & 31))
          tma_load_5d(smem + C::OFF_V + st * C::TILE, &tm_v, &bar_full[st], 0, kt * 128, h, s, b);
      }
      issued = i + 1;
    }
    if (!ok && lane == 0) {
      volatile int no_abort = 0;
      for (int i = max(0, issued - C::NST); i < issued; ++i)
        mbar_wait(&bar_full[i % C::NST], (i / C::NST) & 1, &no_abort);
      mbar_wait(&bar_bias, 0, &no_abort);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ============================ MMA issuer ===============================
    // whole warp, elected lane issues (as in the dK/dV kernel)
    {
      constexpr uint32_t id = idesc_bf16(128, 128, 0, 0);
      // bias tile as the B operand (N = keys, K = queries j'), as in the forward
      constexpr uint32_t id_b = idesc_bf16(128, 128, 0, BIAS_K_CONTIG ? 1 : 0);
      const uint64_t dq0 = umma_desc(smem_u32(smem + C::OFF_Q), 16, C::ATOM, C::SW);
      const uint64_t ddo0 = umma_desc(smem_u32(smem + C::OFF_DO), 16, C::ATOM, C::SW);
      const uint64_t dk0 = umma_desc(smem_u32(smem + C::OFF_K), 16, C::ATOM, C::SW);
      const uint64_t dv0 = umma_desc(smem_u32(smem + C::OFF_V), 16, C::ATOM, C::SW);
      const uint64_t dz0 = umma_desc(smem_u32(smem + C::OFF_Z), 16, 256, kSw32);
      const uint64_t db = BIAS_K_CONTIG
                              ? umma_desc(smem_u32(smem + C::OFF_BIAS), 16384, 1024, kSw128)
                              : umma_desc(smem_u32(smem + C::OFF_BIAS), 16, 1024, kSw128);
      bool ok = __all_sync(0xffffffffu, mbar_wait(&bar_bias, 0, wctx));
      for (int i = 0; i < ns && ok; ++i) {
        const int st = i % C::NST;
        ok = mbar_wait(&bar_full[st], (i / C::NST) & 1, wctx);
        if (ok && i >= 2) ok = mbar_wait(&bar_sdp_free[i & 1], ((i >> 1) - 1) & 1, wctx);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const uint32_t off = (uint32_t)(st * C::TILE) >> 4;
        const uint32_t tsb = tmem + C::T_BUF * (i & 1);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          if (elect_one()) umma_ss(tsb, dq0 + off + 2 * kk, dk0 + off + 2 * kk, id, kk > 0);
          if (elect_one()) umma_ss(tsb + C::T_DP, ddo0 + off + 2 * kk, dv0 + off + 2 * kk, id, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t a = dz0 + ((uint32_t)((112 - 16 * kk) * 32) >> 4);
          const uint64_t bb = BIAS_K_CONTIG
                                  ? db + ((uint32_t)(kk * 2048) >> 4)
                                  : db + ((uint32_t)((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
          if (elect_one()) umma_ss(tsb, a, bb, id_b, 1u);
        }
        if (elect_one()) {
          umma_commit(&bar_empty[st]);
          umma_commit(&bar_s_full[i & 1]);
        }
        __syncwarp();
      }
      if (elect_one()) umma_commit(&bar_drain);
      __syncwarp();
      if (lane == 0) {
        volatile int no_abort = 0;
        mbar_wait(&bar_drain, 0, &no_abort);
      }
    }
    __syncwarp();
  }
  // warps 2-3 have no role
  teardown();
  } else {
    // ============================ compute ==================================
    regs_inc<C::REGS_HIGH>();
    const int wg = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int jl = quad * 32 + lane;
    const int jg = jt * 128 + jl;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    const float c1 = kLog2e * rsqrtf((float)D);
    const float2 c1c1 = make_float2(c1, c1);
    bool ok = true;
    if (p.wc.stall) ok = __all_sync(0xffffffffu, stall_wait(&bar_never, wctx));
    // dbias accumulators of this thread's KPT keys, in registers across all s
    float2 acc[C::KPT / 2];
#pragma unroll
    for (int e = 0; e < C::KPT / 2; ++e) acc[e] = make_float2(0.f, 0.f);
    // lse and delta of the next s are loaded while the current one computes
    float pre_l = 0.f, pre_d = 0.f;
    auto prefetch = [&](int i) {
      if (i >= ns || jg >= p.N) return;
      const int64_t row = (((int64_t)b * p.S + s_begin + i) * p.H + h) * p.N + jg;
      pre_l = p.lse[row];
      pre_d = p.delta[row];
    };
    prefetch(0);
    for (int i = 0; i < ns && ok; ++i) {
      const int st = i % C::NST;
      const float nlse2 = jg < p.N ? -pre_l * kLog2e : -INFINITY;
      const float ndl = jg < p.N ? -pre_d : 0.f;
      prefetch(i + 1);
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_s_full[i & 1], (i >> 1) & 1, wctx));
      if (!ok) break;
      tc_fence_after();
      const float2 nl = make_float2(nlse2, nlse2), nd = make_float2(ndl, ndl);
      const float* madd = reinterpret_cast<const float*>(smem + C::OFF_MADD + st * 512);
      // warp-uniform: most key tiles have no masked key
      const bool masked = *reinterpret_cast<const int*>(smem + C::OFF_FLAG + st * 16) != 0;
#pragma unroll
      for (int q = 0; q < C::KPT / C::CH; ++q) {
        uint32_t sx[C::CH], dpx[C::CH];
        const uint32_t tb = lane_base + C::T_BUF * (i & 1);
        const int k0 = C::KPT * wg + C::CH * q;  // first key of this chunk
        if constexpr (C::CH == 32) {
          tmem_ld32(tb + C::T_S + k0, sx);
          tmem_ld32(tb + C::T_DP + k0, dpx);
        } else {
          tmem_ld16(tb + C::T_S + k0, sx);
          tmem_ld16(tb + C::T_DP + k0, dpx);
        }
        tmem_wait_ld();
        if (q == C::KPT / C::CH - 1) {  // S and dP of this s are in registers
          tc_fence_before();
          mbar_arrive(&bar_sdp_free[i & 1]);
        }
#pragma unroll
        for (int c = 0; c < C::CH / 8; ++c) {
          const int kc = k0 + 8 * c;  // keys kc .. kc + 7
          float2 mv[4];
          if (masked) {
            const float4 ma = *reinterpret_cast<const float4*>(madd + kc);
            const float4 mb = *reinterpret_cast<const float4*>(madd + kc + 4);
            mv[0] = add2(make_float2(ma.x, ma.y), nl); mv[1] = add2(make_float2(ma.z, ma.w), nl);
            mv[2] = add2(make_float2(mb.x, mb.y), nl); mv[3] = add2(make_float2(mb.z, mb.w), nl);
          } else {
            mv[0] = nl; mv[1] = nl; mv[2] = nl; mv[3] = nl;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k2 = 8 * c + 2 * e;
            // S already holds the pair bias (scaled by c = bf16(sqrt(D)))
            const float2 t =
                fma2(make_float2(__uint_as_float(sx[k2]), __uint_as_float(sx[k2 + 1])), c1c1, mv[e]);
            const float2 pr = make_float2(ex2(t.x), ex2(t.y));
            const float2 gg =
                add2(make_float2(__uint_as_float(dpx[k2]), __uint_as_float(dpx[k2 + 1])), nd);
            acc[C::CH / 2 * q + 4 * c + e] = fma2(pr, gg, acc[C::CH / 2 * q + 4 * c + e]);
          }
        }
      }
      mbar_arrive(&bar_empty[st]);
    }
    // ---- write this slot's partial (or add it atomically) ------------------
    if (ok && ns > 0 && jg < p.N) {
      const int64_t base = ((int64_t)b * p.H + h) * p.N * p.N + (int64_t)jg * p.N;
      float* dst = p.atomic ? p.out + base : p.out + (int64_t)slot * p.B * p.H * p.N * p.N + base;
#pragma unroll
      for (int hh = 0; hh < C::KPT / 32; ++hh) {
        const int k0 = kt * 128 + C::KPT * wg + 32 * hh;
        const float2* a2 = acc + 16 * hh;
        if (k0 + 32 <= p.N && (p.N & 3) == 0) {
#pragma unroll
          for (int c = 0; c < 16; c += 2) {
            if (p.atomic)
              red_add_v4(dst + k0 + 2 * c, a2[c].x, a2[c].y, a2[c + 1].x, a2[c + 1].y);
            else
              *reinterpret_cast<float4*>(dst + k0 + 2 * c) =
                  make_float4(a2[c].x, a2[c].y, a2[c + 1].x, a2[c + 1].y);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            if (k0 + 2 * c < p.N) {
              if (p.atomic) atomicAdd(dst + k0 + 2 * c, a2[c].x);
              else dst[k0 + 2 * c] = a2[c].x;
            }
            if (k0 + 2 * c + 1 < p.N) {
              if (p.atomic) atomicAdd(dst + k0 + 2 * c + 1, a2[c].y);
              else dst[k0 + 2 * c + 1] = a2[c].y;
            }
          }
        }
      }
    }
    teardown();
  }
}

// ---------------------------------------------------------------------------
// k_reduce: dbias = ordered sum of the slot partials; dq = bf16 of the dQ
// slices summed in key-tile order (one slice unless dQ is deterministic)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_dbias_sum(const float* __restrict__ partial,
                                                   float* __restrict__ dbias, int64_t n,
                                                   int slots) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if ((n & 3) == 0) {
    const int64_t n4 = n >> 2;
    if (i >= n4) return;
    const float4* src = reinterpret_cast<const float4*>(partial);
    float4 acc = src[i];
    for (int sl = 1; sl < slots; ++sl) {
      const float4 v = src[(int64_t)sl * n4 + i];
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    reinterpret_cast<float4*>(dbias)[i] = acc;
  } else {
    if (i >= n) return;
    float acc = partial[i];
    for (int sl = 1; sl < slots; ++sl) acc += partial[(int64_t)sl * n + i];
    dbias[i] = acc;
  }
}

// SLICED: deterministic dQ, `slices` key-tile partials summed in order; the
// plain conversion stays a separate instantiation so that its register
// count (and occupancy) does not pay for the loop
template <int D, bool SLICED>
__global__ void __launch_bounds__(256) k_dq_convert(const float* __restrict__ dq_acc,
                                                    __nv_bfloat16* __restrict__ dq, Strides5 sdq,
                                                    int B, int S, int H, int N, int slices) {
  constexpr int TPR = D / 8;
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t row = t / TPR;
  const int part = (int)(t % TPR);
  if (row >= (int64_t)B * S * H * N) return;
  const int j = (int)(row % N);
  const int h = (int)((row / N) % H);
  const int s = (int)((row / ((int64_t)N * H)) % S);
  const int b = (int)(row / ((int64_t)N * H * S));
  const float4* src = reinterpret_cast<const float4*>(dq_acc + row * D + 8 * part);
  float4 a = src[0], c = src[1];
  if (SLICED) {
    const int64_t slice4 = (int64_t)B * S * H * N * (D / 4);
    for (int k = 1; k < slices; ++k) {
      const float4 x = src[k * slice4], y = src[k * slice4 + 1];
      a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
      c.x += y.x; c.y += y.y; c.z += y.z; c.w += y.w;
    }
  }
  const float f[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
  *reinterpret_cast<uint4*>(dq + sdq.at(b, s, h, j, 8 * part)) = pack8(f);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
bool tmap_rows(CUtensorMap* m, const void* base, const Strides5& st, const Problem& P) {
  const uint64_t dims[5] = {(uint64_t)P.D, (uint64_t)P.N, (uint64_t)P.H, (uint64_t)P.S,
                            (uint64_t)P.B};
  const uint64_t str[4] = {(uint64_t)st.n * 2, (uint64_t)st.h * 2, (uint64_t)st.s * 2,
                           (uint64_t)st.b * 2};
  const uint32_t box[5] = {(uint32_t)P.D, 128, 1, 1, 1};
  const CUtensorMapSwizzle sw =
      P.D == 16 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B;
  // No L2 promotion: a box row is D * 2 = 32 or 64 bytes, and in the
  // ending-node layout ([B, N_i, N_j, H, D] read with s = j) the rest of a
  // 256-byte line is the other heads' rows, which k_dbias's CTAs (heads in
  // different waves) do not use while the line is in L2.  Measured on the
  // N = 768 ending-node workload: k_dbias DRAM reads 1.55 -> 1.27 GB, times
  // unchanged.
  return make_tmap_bf16(m, base, 5, dims, str, box, sw, CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

bool tmap_bias(CUtensorMap* m, const void* base, const StridesBias& sb, const Problem& P,
               bool k_contig) {
  const uint64_t dims[4] = {(uint64_t)P.N, (uint64_t)P.N, (uint64_t)P.H, (uint64_t)P.B};
  const uint64_t outer = k_contig ? sb.j : sb.k;
  const uint64_t str[3] = {outer * 2, (uint64_t)sb.h * 2, (uint64_t)sb.b * 2};
  const uint32_t box[4] = {64, 128, 1, 1};
  return make_tmap_bf16(m, base, 4, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <typename K>
cudaError_t set_smem(K kern, uint32_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// A kernel that splits registers between warpgroups (setmaxnreg) must be
// launched with at least the per-thread count the split was sized for, or its
// raising warpgroups would wait forever: refuse to launch otherwise.
template <typename K>
cudaError_t check_regs(K kern, int launch_regs) {
  cudaFuncAttributes fa{};
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  return fa.numRegs >= launch_regs ? cudaSuccess : cudaErrorInvalidConfiguration;
}

template <int D, bool KC>
cudaError_t bwd_launch(const Problem& P, const Bf16Ptrs& a, unsigned flags, const Workspace& w,
                       const WaitCfg& wait, cudaStream_t st, const CUtensorMap& tq,
                       const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                       const CUtensorMap& tb, const Strides5& ado, const PreParams& walk,
                       cudaEvent_t* ev) {
  const int nt = (P.N + 127) / 128;
  if (ev) cudaEventRecord(ev[0], st);
  // 1) delta, dgate, dOa; zero dQ accumulator
  {
    PreParams pp = walk;
    pp.B = P.B; pp.S = P.S; pp.H = P.H; pp.N = P.N; pp.D = D;
    pp.a = ado;
    pp.out = static_cast<const __nv_bfloat16*>(a.out);
    pp.dout = static_cast<const __nv_bfloat16*>(a.dout);
    pp.gate = static_cast<const __nv_bfloat16*>(a.gate);
    pp.o = P.o; pp.dO = P.dout; pp.g = P.g; pp.dg = P.dg;
    pp.dgate = static_cast<__nv_bfloat16*>(a.dgate);
    pp.dOa = w.dOa; pp.delta = w.delta;
    pp.dq_acc = w.dq_slices == 1 ? w.dq_acc : nullptr;  // slices are stored, not added to
    constexpr int U = 2;
    const int64_t units = P.rows() * (D / 8);
    k_pre<D, U><<<(unsigned)((units + 256 * U - 1) / (256 * U)), 256, 0, st>>>(pp);
  }
  const bool fused = (flags & EVOATTN_DBIAS_FUSED) != 0;
  if (fused || (flags & EVOATTN_DBIAS_ATOMIC)) {
    cudaError_t e = cudaMemsetAsync(a.dbias, 0, (size_t)P.B * P.H * P.N * P.N * 4, st);
    if (e != cudaSuccess) return e;
  }
  if (ev) cudaEventRecord(ev[1], st);
  // 2) dK, dV (+ dQ partial sums)
  {
    using C = DkdvCfg<D, KC>;
    DkdvParams dp{};
    dp.B = P.B; dp.S = P.S; dp.H = P.H; dp.N = P.N; dp.njt = nt; dp.nkt = nt;
    const int64_t items = (int64_t)P.B * P.S * P.H * nt;
    if (items > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    dp.n_items = (int)items;
    dp.mask = a.mask; dp.msb = P.mask.b; dp.mss = P.mask.s; dp.msk = P.mask.k;
    dp.lse = a.lse; dp.delta = w.delta; dp.dq_acc = w.dq_acc;
    dp.dq_det = w.dq_slices > 1 ? 1 : 0;
    dp.dq_slice = P.rows() * D;
    dp.dk = static_cast<__nv_bfloat16*>(a.dk); dp.dv = static_cast<__nv_bfloat16*>(a.dv);
    dp.sdk = P.dk; dp.sdv = P.dv; dp.wc = launch_wait(wait);
    dp.dbias = static_cast<float*>(a.dbias);
    auto kern = fused ? k_dkdv<D, KC, true> : k_dkdv<D, KC, false>;
    cudaError_t e = set_smem(kern, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    e = check_regs(kern, C::LAUNCH_REGS);
    if (e != cudaSuccess) return e;
    // persistent: one CTA per SM (each holds 512 TMEM columns)
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int grid = (int)std::min<int64_t>(items, (int64_t)std::max(sms, 1));
    kern<<<grid, C::THREADS, C::SMEM_ALLOC, st>>>(tq, tk, tv, tdo, tb, dp);
  }
  if (ev) cudaEventRecord(ev[2], st);
  // 3) dbias partials (none when dbias was summed in step 2)
  const int slots = dbias_slots(P);
  if (!fused) {
    using C = DbiasCfg<D>;
    DbiasParams bp{};
    bp.B = P.B; bp.S = P.S; bp.H = P.H; bp.N = P.N; bp.njt = nt; bp.nkt = nt;
    bp.slots = slots;
    bp.mask = a.mask; bp.msb = P.mask.b; bp.mss = P.mask.s; bp.msk = P.mask.k;
    bp.lse = a.lse; bp.delta = w.delta;
    bp.atomic = (flags & EVOATTN_DBIAS_ATOMIC) ? 1 : 0;
    bp.out = bp.atomic ? a.dbias : w.partial;
    bp.wc = launch_wait(wait);
    auto kern = k_dbias<D, KC>;
    cudaError_t e = set_smem(kern, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    e = check_regs(kern, C::LAUNCH_REGS);
    if (e != cudaSuccess) return e;
    const uint64_t grid = (uint64_t)P.B * P.H * slots * nt * nt;
    if (grid > 0x7FFFFFFFull) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)grid, C::THREADS, C::SMEM_ALLOC, st>>>(tq, tk, tv, tdo, tb, bp);
  }
  if (ev) cudaEventRecord(ev[3], st);
  // 4) ordered slot sum, dQ conversion
  if (!fused && !(flags & EVOATTN_DBIAS_ATOMIC)) {
    const int64_t n = (int64_t)P.B * P.H * P.N * P.N;
    const int64_t work = (n & 3) == 0 ? n / 4 : n;
    k_dbias_sum<<<(unsigned)((work + 255) / 256), 256, 0, st>>>(w.partial, a.dbias, n, slots);
  }
  {
    const int64_t threads = P.rows() * (D / 8);
    const unsigned blocks = (unsigned)((threads + 255) / 256);
    if (w.dq_slices > 1)
      k_dq_convert<D, true><<<blocks, 256, 0, st>>>(
          w.dq_acc, static_cast<__nv_bfloat16*>(a.dq), P.dq, P.B, P.S, P.H, P.N, w.dq_slices);
    else
      k_dq_convert<D, false><<<blocks, 256, 0, st>>>(
          w.dq_acc, static_cast<__nv_bfloat16*>(a.dq), P.dq, P.B, P.S, P.H, P.N, 1);
  }
  if (ev) cudaEventRecord(ev[4], st);
  return cudaGetLastError();
}

template <int D>
cudaError_t bwd_d(const Problem& P, const Bf16Ptrs& a, unsigned flags, void* ws,
                  const WaitCfg& wait, cudaStream_t st, bool* tmap_ok, cudaEvent_t* ev) {
  const Workspace w = carve(P, flags, ws);
  // dOa is dense in the memory order of out
  PreParams walk{};
  const Strides5 ado = dense_like(P, P.o, walk.walk_dim, walk.walk_size);
  CUtensorMap tq, tk, tv, tdo, tb;
  const bool kc = P.bias.k == 1;
  if (!tmap_rows(&tq, a.q, P.q, P) || !tmap_rows(&tk, a.k, P.k, P) ||
      !tmap_rows(&tv, a.v, P.v, P) || !tmap_rows(&tdo, w.dOa, ado, P) ||
      !tmap_bias(&tb, a.bias, P.bias, P, kc)) {
    *tmap_ok = false;
    return cudaErrorInvalidValue;
  }
  return kc ? bwd_launch<D, true>(P, a, flags, w, wait, st, tq, tk, tv, tdo, tb, ado, walk, ev)
            : bwd_launch<D, false>(P, a, flags, w, wait, st, tq, tk, tv, tdo, tb, ado, walk, ev);
}

}  // namespace

size_t bf16_bwd_workspace_bytes(const Problem& P, unsigned flags) {
  if (P.D != 16 && P.D != 32) return 0;
  return carve(P, flags, nullptr).bytes;
}

cudaError_t bf16_bwd(const Problem& P, const Bf16Ptrs& a, unsigned flags, void* ws,
                     const WaitCfg& wait, cudaStream_t st, bool* tmap_ok,
                     cudaEvent_t* events) {
  switch (P.D) {
    case 16: return bwd_d<16>(P, a, flags, ws, wait, st, tmap_ok, events);
    case 32: return bwd_d<32>(P, a, flags, ws, wait, st, tmap_ok, events);
  }
  return cudaErrorNotSupported;
}

}  // namespace evo
