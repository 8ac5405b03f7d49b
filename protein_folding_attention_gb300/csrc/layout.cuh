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

// The additive logit offset that a masked key receives.
constexpr float kMaskBias = -1.0e9f;

}  // namespace evo
