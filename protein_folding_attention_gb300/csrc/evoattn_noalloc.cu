// evoattn_bwd_noalloc: the backward with library-owned scratch, for callers
// that cannot allocate device memory (see include/evoattn.h).
#include <cuda_runtime.h>

#include <mutex>

#include "evoattn.h"

namespace {

// The scratch: one fixed-size array per device, held for the life of the
// process.  In host code `g_noalloc_scratch` names a host-side stand-in, not
// device memory; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[EVOATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of the scratch array on the current device, looked up once
// per device with that device current.  Returns nullptr on failure.
void* scratch_address() {
  static void* addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" evoattn_status evoattn_bwd_noalloc(
    const void* q, const int64_t q_strides[5], const void* k, const int64_t k_strides[5],
    const void* v, const int64_t v_strides[5], const void* pair_bias,
    const int64_t bias_strides[4], const uint8_t* mask, const int64_t mask_strides[3],
    const void* gate, const int64_t gate_strides[5], const void* out,
    const int64_t out_strides[5], const float* lse, const void* dout,
    const int64_t dout_strides[5], void* dq, const int64_t dq_strides[5], void* dk,
    const int64_t dk_strides[5], void* dv, const int64_t dv_strides[5], float* dbias,
    void* dgate, const int64_t dgate_strides[5], int B, int S, int H, int N, int D,
    evoattn_dtype dtype, unsigned flags, cudaStream_t stream) {
  const size_t need = evoattn_bwd_workspace_size(B, S, H, N, D, dtype, flags);
  if (need == 0)  // sizes, D, dtype or flags invalid: let the checks name the error
    return evoattn_bwd(q, q_strides, k, k_strides, v, v_strides, pair_bias, bias_strides,
                       mask, mask_strides, gate, gate_strides, out, out_strides, lse, dout,
                       dout_strides, dq, dq_strides, dk, dk_strides, dv, dv_strides, dbias,
                       dgate, dgate_strides, B, S, H, N, D, dtype, flags, nullptr, 0, stream);
  if (need > EVOATTN_NOALLOC_SCRATCH_BYTES) return EVOATTN_ERR_WORKSPACE;
  void* scratch = scratch_address();
  if (!scratch) return EVOATTN_ERR_CUDA;
  return evoattn_bwd(q, q_strides, k, k_strides, v, v_strides, pair_bias, bias_strides, mask,
                     mask_strides, gate, gate_strides, out, out_strides, lse, dout,
                     dout_strides, dq, dq_strides, dk, dk_strides, dv, dv_strides, dbias, dgate,
                     dgate_strides, B, S, H, N, D, dtype, flags, scratch,
                     EVOATTN_NOALLOC_SCRATCH_BYTES, stream);
}
