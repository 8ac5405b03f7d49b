// FP32 per-row kernels (see simt_f32.cu).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>

#include "layout.cuh"

namespace evo {

struct F32Ptrs {
  const float *q, *k, *v, *bias, *gate, *dout;
  const unsigned char* mask;
  float* out;  // forward: written; backward: read
  float* lse;  // forward: written; backward: read
  float *dq, *dk, *dv, *dbias, *dgate;
};

size_t f32_bwd_workspace_bytes(const Problem& P);
cudaError_t f32_fwd(const Problem& P, const F32Ptrs& a, cudaStream_t st);
cudaError_t f32_bwd(const Problem& P, const F32Ptrs& a, void* ws, cudaStream_t st,
                    cudaEvent_t* events);

}  // namespace evo
