// Problem description shared by the host launcher and the kernels: sizes and
// element strides of every operand (logical shapes as in evoattn.h).
#pragma once
#include <stdint.h>

namespace evo {

struct Strides5 {
  int64_t b, s, h, n, d;
  __host__ __device__ int64_t at(int64_t bb, int64_t ss, int64_t hh, int64_t nn,
                                 int64_t dd) const {
    return bb * b + ss * s + hh * h + nn * n + dd * d;
  }
};
struct StridesBias {
  int64_t b, h, j, k;
  __host__ __device__ int64_t at(int64_t bb, int64_t hh, int64_t jj, int64_t kk) const {
    return bb * b + hh * h + jj * j + kk * k;
  }
};
struct StridesMask {
  int64_t b, s, k;
  __host__ __device__ int64_t at(int64_t bb, int64_t ss, int64_t kk) const {
    return bb * b + ss * s + kk * k;
  }
};

struct Problem {
  int B, S, H, N, D;
  Strides5 q, k, v, g, o, dout, dq, dk, dv, dg;
  StridesBias bias;
  StridesMask mask;
  // Rows are (b,s,h,n) in this order; row r of a dense [B,S,H,N] array.
  __host__ __device__ int64_t rows() const { return (int64_t)B * S * H * N; }
};

// Default limit of a pipeline wait, in nanoseconds of %globaltimer time.  The
// waits of the wind-down after a give-up always use this limit.
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // 2 s

// Per-launch configuration of the bounded waits of a tcgen05 kernel, passed
// by value in its parameters (see common.cuh).
struct WaitCfg {
  unsigned int* status;         // device words: [0] status bits, [1] abort word
  unsigned int launch;          // this launch's id (never 0)
  int stall;                    // testing: the compute warps' first wait never completes
  unsigned long long limit_ns;  // limit of every pipeline wait
};

// The additive logit offset that a masked key receives.
constexpr float kMaskBias = -1.0e9f;

}  // namespace evo
