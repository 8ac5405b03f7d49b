// Launchers of the tcgen05/TMA (sm_103a) kernels of the BF16 path.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

#include "layout.cuh"

namespace evo {

struct Bf16Ptrs {
  const void *q, *k, *v, *bias, *gate, *dout;
  const unsigned char* mask;
  void* out;   // forward: written; backward: read
  float* lse;  // forward: written; backward: read
  void *dq, *dk, *dv, *dgate;
  float* dbias;
};

// A fresh id for the next kernel launch (never 0).
unsigned int next_launch_id();

// The wait configuration of one launch: `base` with a fresh launch id.
inline WaitCfg launch_wait(const WaitCfg& base) {
  WaitCfg c = base;
  c.launch = next_launch_id();
  return c;
}

// Returns cudaSuccess or the first launch / tensor-map error.  `wait` holds
// the device status words and the wait limit (its launch id is replaced per
// launch).  `tmap_ok` is set false when the driver rejected a tensor map
// (alignment or size).
cudaError_t bf16_fwd(const Problem& P, const Bf16Ptrs& a, const WaitCfg& wait,
                     cudaStream_t st, bool* tmap_ok);

// LayerNorm + projection (EvoFusion upstream); C = 128 and H * D = 128.
cudaError_t bf16_ln_proj(const void* z, const float* gamma, const float* beta, const void* w,
                         float eps, void* q, void* k, void* v, void* g, void* bias, int B, int N,
                         int H, const WaitCfg& wait, cudaStream_t st, bool* tmap_ok);

// Output projection (o and w_o nullable together) + SwiGLU transition
// (EvoFusion downstream); C = 128, H * D = 128, F = 4C.
cudaError_t bf16_transition(const void* z, const void* o, const void* w_o, const float* gamma,
                            const float* beta, const void* w1, const void* w2, float eps,
                            void* out, int B, int N, const WaitCfg& wait, cudaStream_t st,
                            bool* tmap_ok);

size_t bf16_bwd_workspace_bytes(const Problem& P, unsigned flags);
// `events` (nullable): 5 caller-owned events recorded around the stages.
cudaError_t bf16_bwd(const Problem& P, const Bf16Ptrs& a, unsigned flags, void* ws,
                     const WaitCfg& wait, cudaStream_t st, bool* tmap_ok,
                     cudaEvent_t* events);

}  // namespace evo
