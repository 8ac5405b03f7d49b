// FP32 path: plain per-row CUDA kernels in single precision.
//
// The tensor-core path computes in bf16 with fp32 accumulation, which cannot
// meet a 1e-5 relative tolerance; fp32 inputs therefore run these kernels,
// which keep every product and sum in fp32.  One thread owns one query row
// (forward, dq), one key (dk/dv) or one bias entry (dbias), so every result is
// a fixed-order sum and the whole backward is deterministic.  They compute
// the same expression as the tensor-core kernels (MegaFold technical summary,
// "Methodik" section 1 "EvoFlash-3D": online numerically stable softmax over
// pair-biased logits) without tiling; they are meant for small problems.
#include <cuda_runtime.h>
#include <math.h>

#include "layout.cuh"
#include "simt_f32.h"

namespace evo {
namespace {

__device__ __forceinline__ float sigm(float x) { return 1.0f / (1.0f + expf(-x)); }

// logit of (b,s,h,j,k) from an already loaded query row.
template <int D>
__device__ __forceinline__ float logit(const Problem& P, const float* __restrict__ k,
                                       const float* __restrict__ bias,
                                       const unsigned char* __restrict__ mask,
                                       const float (&qj)[D], int b, int s, int h, int j,
                                       int kk, float scale) {
  const float* kr = k + P.k.at(b, s, h, kk, 0);
  float dot = 0.f;
#pragma unroll
  for (int d = 0; d < D; ++d) dot = fmaf(qj[d], kr[d * P.k.d], dot);
  float x = dot * scale + bias[P.bias.at(b, h, j, kk)];
  if (mask && !mask[P.mask.at(b, s, kk)]) x += kMaskBias;
  return x;
}

template <int D>
__global__ void fwd_f32_kernel(Problem P, const float* __restrict__ q,
                               const float* __restrict__ k, const float* __restrict__ v,
                               const float* __restrict__ bias,
                               const unsigned char* __restrict__ mask,
                               const float* __restrict__ gate, float* __restrict__ out,
                               float* __restrict__ lse) {
  const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= P.rows()) return;
  const int j = (int)(row % P.N);
  const int h = (int)((row / P.N) % P.H);
  const int s = (int)((row / ((int64_t)P.N * P.H)) % P.S);
  const int b = (int)(row / ((int64_t)P.N * P.H * P.S));
  const float scale = rsqrtf((float)D);
  float qj[D], acc[D];
#pragma unroll
  for (int d = 0; d < D; ++d) {
    qj[d] = q[P.q.at(b, s, h, j, d)];
    acc[d] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int kk = 0; kk < P.N; ++kk) {
    const float x = logit<D>(P, k, bias, mask, qj, b, s, h, j, kk, scale);
    const float m_new = fmaxf(m, x);
    const float alpha = expf(m - m_new);  // 0 on the first key
    const float p = expf(x - m_new);
    l = l * alpha + p;
    const float* vr = v + P.v.at(b, s, h, kk, 0);
#pragma unroll
    for (int d = 0; d < D; ++d) acc[d] = fmaf(p, vr[d * P.v.d], acc[d] * alpha);
    m = m_new;
  }
  const float inv_l = 1.0f / l;
#pragma unroll
  for (int d = 0; d < D; ++d) {
    float o = acc[d] * inv_l;
    if (gate) o *= sigm(gate[P.g.at(b, s, h, j, d)]);
    out[P.o.at(b, s, h, j, d)] = o;
  }
  lse[row] = m + logf(l);
}

// delta = sum_d dout*out, dgate = dout*out*(1-sigmoid(g)), dOa = dout*sigmoid(g)
template <int D>
__global__ void bwd_pre_f32_kernel(Problem P, const float* __restrict__ out,
                                   const float* __restrict__ dout,
                                   const float* __restrict__ gate, float* __restrict__ dgate,
                                   float* __restrict__ dOa, float* __restrict__ delta) {
  const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= P.rows()) return;
  const int j = (int)(row % P.N);
  const int h = (int)((row / P.N) % P.H);
  const int s = (int)((row / ((int64_t)P.N * P.H)) % P.S);
  const int b = (int)(row / ((int64_t)P.N * P.H * P.S));
  float dl = 0.f;
#pragma unroll
  for (int d = 0; d < D; ++d) {
    const float o = out[P.o.at(b, s, h, j, d)];
    const float go = dout[P.dout.at(b, s, h, j, d)];
    dl = fmaf(go, o, dl);
    float sg = 1.f;
    if (gate) {
      sg = sigm(gate[P.g.at(b, s, h, j, d)]);
      dgate[P.dg.at(b, s, h, j, d)] = go * o * (1.f - sg);
    }
    dOa[row * D + d] = go * sg;
  }
  delta[row] = dl;
}

template <int D>
__global__ void bwd_dq_f32_kernel(Problem P, const float* __restrict__ q,
                                  const float* __restrict__ k, const float* __restrict__ v,
                                  const float* __restrict__ bias,
                                  const unsigned char* __restrict__ mask,
                                  const float* __restrict__ lse, const float* __restrict__ dOa,
                                  const float* __restrict__ delta, float* __restrict__ dq) {
  const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= P.rows()) return;
  const int j = (int)(row % P.N);
  const int h = (int)((row / P.N) % P.H);
  const int s = (int)((row / ((int64_t)P.N * P.H)) % P.S);
  const int b = (int)(row / ((int64_t)P.N * P.H * P.S));
  const float scale = rsqrtf((float)D);
  float qj[D], go[D], acc[D];
#pragma unroll
  for (int d = 0; d < D; ++d) {
    qj[d] = q[P.q.at(b, s, h, j, d)];
    go[d] = dOa[row * D + d];
    acc[d] = 0.f;
  }
  const float L = lse[row], dl = delta[row];
  for (int kk = 0; kk < P.N; ++kk) {
    const float p = expf(logit<D>(P, k, bias, mask, qj, b, s, h, j, kk, scale) - L);
    const float* vr = v + P.v.at(b, s, h, kk, 0);
    float dp = 0.f;
#pragma unroll
    for (int d = 0; d < D; ++d) dp = fmaf(go[d], vr[d * P.v.d], dp);
    const float ds = p * (dp - dl);
    const float* kr = k + P.k.at(b, s, h, kk, 0);
#pragma unroll
    for (int d = 0; d < D; ++d) acc[d] = fmaf(ds, kr[d * P.k.d], acc[d]);
  }
#pragma unroll
  for (int d = 0; d < D; ++d) dq[P.dq.at(b, s, h, j, d)] = acc[d] * scale;
}

template <int D>
__global__ void bwd_dkdv_f32_kernel(Problem P, const float* __restrict__ q,
                                    const float* __restrict__ k, const float* __restrict__ v,
                                    const float* __restrict__ bias,
                                    const unsigned char* __restrict__ mask,
                                    const float* __restrict__ lse,
                                    const float* __restrict__ dOa,
                                    const float* __restrict__ delta, float* __restrict__ dk,
                                    float* __restrict__ dv) {
  const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // (b,s,h,key)
  if (row >= P.rows()) return;
  const int kk = (int)(row % P.N);
  const int h = (int)((row / P.N) % P.H);
  const int s = (int)((row / ((int64_t)P.N * P.H)) % P.S);
  const int b = (int)(row / ((int64_t)P.N * P.H * P.S));
  const float scale = rsqrtf((float)D);
  const int64_t row0 = row - kk;  // row index of (b,s,h,0)
  float kr[D], vr[D], adk[D], adv[D];
#pragma unroll
  for (int d = 0; d < D; ++d) {
    kr[d] = k[P.k.at(b, s, h, kk, d)];
    vr[d] = v[P.v.at(b, s, h, kk, d)];
    adk[d] = 0.f;
    adv[d] = 0.f;
  }
  const bool keep = !mask || mask[P.mask.at(b, s, kk)];
  for (int j = 0; j < P.N; ++j) {
    const float* qj = q + P.q.at(b, s, h, j, 0);
    float dot = 0.f;
#pragma unroll
    for (int d = 0; d < D; ++d) dot = fmaf(qj[d * P.q.d], kr[d], dot);
    float x = dot * scale + bias[P.bias.at(b, h, j, kk)];
    if (!keep) x += kMaskBias;
    const float p = expf(x - lse[row0 + j]);
    const float* go = dOa + (row0 + j) * D;
    float dp = 0.f;
#pragma unroll
    for (int d = 0; d < D; ++d) dp = fmaf(go[d], vr[d], dp);
    const float ds = p * (dp - delta[row0 + j]);
#pragma unroll
    for (int d = 0; d < D; ++d) {
      adk[d] = fmaf(ds, qj[d * P.q.d], adk[d]);
      adv[d] = fmaf(p, go[d], adv[d]);
    }
  }
#pragma unroll
  for (int d = 0; d < D; ++d) {
    dk[P.dk.at(b, s, h, kk, d)] = adk[d] * scale;
    dv[P.dv.at(b, s, h, kk, d)] = adv[d];
  }
}

// dbias[b,h,j,k] = sum over s (ascending) of ds.
template <int D>
__global__ void bwd_dbias_f32_kernel(Problem P, const float* __restrict__ q,
                                     const float* __restrict__ k, const float* __restrict__ v,
                                     const float* __restrict__ bias,
                                     const unsigned char* __restrict__ mask,
                                     const float* __restrict__ lse,
                                     const float* __restrict__ dOa,
                                     const float* __restrict__ delta,
                                     float* __restrict__ dbias) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // (b,h,j,k)
  const int64_t total = (int64_t)P.B * P.H * P.N * P.N;
  if (e >= total) return;
  const int kk = (int)(e % P.N);
  const int j = (int)((e / P.N) % P.N);
  const int h = (int)((e / ((int64_t)P.N * P.N)) % P.H);
  const int b = (int)(e / ((int64_t)P.N * P.N * P.H));
  const float scale = rsqrtf((float)D);
  const float bj = bias[P.bias.at(b, h, j, kk)];
  float acc = 0.f;
  for (int s = 0; s < P.S; ++s) {
    const float* qj = q + P.q.at(b, s, h, j, 0);
    const float* kr = k + P.k.at(b, s, h, kk, 0);
    const float* vr = v + P.v.at(b, s, h, kk, 0);
    const int64_t row = (((int64_t)b * P.S + s) * P.H + h) * P.N + j;
    const float* go = dOa + row * D;
    float dot = 0.f, dp = 0.f;
#pragma unroll
    for (int d = 0; d < D; ++d) {
      dot = fmaf(qj[d * P.q.d], kr[d * P.k.d], dot);
      dp = fmaf(go[d], vr[d * P.v.d], dp);
    }
    float x = dot * scale + bj;
    if (mask && !mask[P.mask.at(b, s, kk)]) x += kMaskBias;
    const float p = expf(x - lse[row]);
    acc += p * (dp - delta[row]);
  }
  dbias[e] = acc;
}

inline unsigned blocks_for(int64_t n, int t) { return (unsigned)((n + t - 1) / t); }

template <int D>
cudaError_t fwd_f32_d(const Problem& P, const F32Ptrs& a, cudaStream_t st) {
  const int T = 128;
  fwd_f32_kernel<D><<<blocks_for(P.rows(), T), T, 0, st>>>(
      P, a.q, a.k, a.v, a.bias, a.mask, a.gate, a.out, a.lse);
  return cudaGetLastError();
}

template <int D>
cudaError_t bwd_f32_d(const Problem& P, const F32Ptrs& a, float* ws, cudaStream_t st,
                      cudaEvent_t* ev) {
  const int T = 128;
  float* dOa = ws;
  float* delta = ws + P.rows() * D;
  if (ev) cudaEventRecord(ev[0], st);
  bwd_pre_f32_kernel<D><<<blocks_for(P.rows(), T), T, 0, st>>>(P, a.out, a.dout, a.gate,
                                                                a.dgate, dOa, delta);
  if (ev) cudaEventRecord(ev[1], st);
  bwd_dq_f32_kernel<D><<<blocks_for(P.rows(), T), T, 0, st>>>(
      P, a.q, a.k, a.v, a.bias, a.mask, a.lse, dOa, delta, a.dq);
  bwd_dkdv_f32_kernel<D><<<blocks_for(P.rows(), T), T, 0, st>>>(
      P, a.q, a.k, a.v, a.bias, a.mask, a.lse, dOa, delta, a.dk, a.dv);
  if (ev) cudaEventRecord(ev[2], st);
  const int64_t nb = (int64_t)P.B * P.H * P.N * P.N;
  bwd_dbias_f32_kernel<D><<<blocks_for(nb, T), T, 0, st>>>(
      P, a.q, a.k, a.v, a.bias, a.mask, a.lse, dOa, delta, a.dbias);
  if (ev) { cudaEventRecord(ev[3], st); cudaEventRecord(ev[4], st); }
  return cudaGetLastError();
}

}  // namespace

size_t f32_bwd_workspace_bytes(const Problem& P) {
  return (size_t)P.rows() * (P.D + 1) * sizeof(float);
}

cudaError_t f32_fwd(const Problem& P, const F32Ptrs& a, cudaStream_t st) {
  switch (P.D) {
    case 16: return fwd_f32_d<16>(P, a, st);
    case 32: return fwd_f32_d<32>(P, a, st);
    case 64: return fwd_f32_d<64>(P, a, st);
    case 128: return fwd_f32_d<128>(P, a, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t f32_bwd(const Problem& P, const F32Ptrs& a, void* ws, cudaStream_t st,
                    cudaEvent_t* ev) {
  float* w = static_cast<float*>(ws);
  switch (P.D) {
    case 16: return bwd_f32_d<16>(P, a, w, st, ev);
    case 32: return bwd_f32_d<32>(P, a, w, st, ev);
    case 64: return bwd_f32_d<64>(P, a, w, st, ev);
    case 128: return bwd_f32_d<128>(P, a, w, st, ev);
  }
  return cudaErrorInvalidValue;
}

}  // namespace evo
