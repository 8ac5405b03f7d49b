// C ABI of the EvoAttention library: host-side validation and dispatch.
// Every check happens before anything is enqueued; see include/evoattn.h for
// the contract.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "evoattn.h"
#include "layout.cuh"
#include "simt_f32.h"
#include "sm103.h"

namespace evo {

// Two words per device: [0] status bits the kernels OR into (read and cleared
// by evoattn_get_device_status), [1] the id of the latest launch that gave up
// a wait (the other CTAs of that launch poll it).
__device__ unsigned int g_device_status_words[2] = {0u, 0u};

namespace {
std::atomic<unsigned int> g_launch_counter{0};
// testing hook state (evoattn_debug_set_wait)
std::atomic<unsigned long long> g_wait_limit_ns{kWaitTimeoutNs};
std::atomic<int> g_wait_stall{0};
}  // namespace

unsigned int next_launch_id() {
  unsigned int id = ++g_launch_counter;
  if (id == 0) id = ++g_launch_counter;  // 0 never names a launch
  return id;
}

namespace {

constexpr int kMaxDevices = 64;

// Device address of the status words of the current device (looked up once
// per device, with that device current).
unsigned int* status_word(bool* ok) {
  static unsigned int* addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *ok = false;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status_words) != cudaSuccess) {
      *ok = false;
      return nullptr;
    }
    addr[dev] = static_cast<unsigned int*>(p);
  }
  *ok = true;
  return addr[dev];
}

bool d_supported(evoattn_dtype dt, int D) {
  if (dt == EVOATTN_BF16) return D == 16 || D == 32 || D == 64;
  if (dt == EVOATTN_F32) return D == 16 || D == 32 || D == 64 || D == 128;
  return false;
}
// The BF16 backward has D = 16 and D = 32 kernels only.
bool d_supported_bwd(evoattn_dtype dt, int D) {
  if (dt == EVOATTN_BF16) return D == 16 || D == 32;
  return d_supported(dt, D);
}

// Wait configuration of the next launches on the current device.
WaitCfg wait_base(unsigned int* status) {
  WaitCfg w{};
  w.status = status;
  w.launch = 0;
  w.stall = g_wait_stall.load();
  w.limit_ns = g_wait_limit_ns.load();
  return w;
}

bool nonneg(const int64_t* s, int n) {
  for (int i = 0; i < n; ++i)
    if (s[i] < 0) return false;
  return true;
}

Strides5 s5(const int64_t* s) { return Strides5{s[0], s[1], s[2], s[3], s[4]}; }

// BF16 tensor-core path: unit d stride, 16-byte aligned base and strides.
bool bf16_ok5(const void* p, const int64_t* s) {
  if (!p) return true;
  if (reinterpret_cast<uintptr_t>(p) % 16) return false;
  if (s[4] != 1) return false;
  for (int i = 0; i < 4; ++i)
    if (s[i] % 8) return false;
  return true;
}
bool bf16_ok_bias(const void* p, const int64_t* s) {
  if (reinterpret_cast<uintptr_t>(p) % 16) return false;
  // {b, h, j, k}: unit stride along k (j stride aligned) or along j (k stride aligned)
  if (s[0] % 8 || s[1] % 8) return false;
  if (s[3] == 1) return s[2] % 8 == 0;
  if (s[2] == 1) return s[3] % 8 == 0;
  return false;
}

evoattn_status cuda_status(cudaError_t e) { return e == cudaSuccess ? EVOATTN_OK : EVOATTN_ERR_CUDA; }

}  // namespace
}  // namespace evo

using namespace evo;

extern "C" {

int evoattn_version(void) { return 200; }  // 0.2.0

evoattn_status evoattn_debug_set_wait(unsigned long long limit_ns, int stall) {
  g_wait_limit_ns.store(limit_ns == 0 ? kWaitTimeoutNs : limit_ns);
  g_wait_stall.store(stall != 0 ? 1 : 0);
  return EVOATTN_OK;
}

const char* evoattn_status_string(evoattn_status s) {
  switch (s) {
    case EVOATTN_OK: return "ok";
    case EVOATTN_ERR_INVALID_ARG: return "invalid argument (null pointer, size or flag)";
    case EVOATTN_ERR_UNSUPPORTED: return "unsupported dtype or head dimension";
    case EVOATTN_ERR_ALIGNMENT: return "stride or address breaks the BF16 alignment rules";
    case EVOATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case EVOATTN_ERR_CUDA: return "CUDA runtime or driver call failed";
    case EVOATTN_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
  }
  return "unknown status";
}

evoattn_status evoattn_ln_proj(const void* z, const float* gamma, const float* beta,
                               const void* w, float eps, void* q, void* k, void* v, void* g,
                               void* pair_bias, int B, int N, int C, int H, int D,
                               cudaStream_t stream) {
  if (!z || !gamma || !beta || !w || !q || !k || !v || !g || !pair_bias)
    return EVOATTN_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || C < 1 || H < 1 || D < 1) return EVOATTN_ERR_INVALID_ARG;
  if (!(eps > 0.f) || !(eps < INFINITY)) return EVOATTN_ERR_INVALID_ARG;
  if (C != 128 || H * D != 128 || H > 8) return EVOATTN_ERR_UNSUPPORTED;
  if ((uint64_t)B * N * N + 128 > 0x7FFFFFFFull) return EVOATTN_ERR_UNSUPPORTED;
  auto a16 = [](const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; };
  if (!a16(z) || !a16(w) || !a16(q) || !a16(k) || !a16(v) || !a16(g) ||
      reinterpret_cast<uintptr_t>(gamma) % 4 || reinterpret_cast<uintptr_t>(beta) % 4 ||
      reinterpret_cast<uintptr_t>(pair_bias) % 2)
    return EVOATTN_ERR_ALIGNMENT;
  bool ok = false;
  unsigned int* status = status_word(&ok);
  if (!ok) return EVOATTN_ERR_CUDA;
  bool tmap_ok = true;
  cudaError_t e = bf16_ln_proj(z, gamma, beta, w, eps, q, k, v, g, pair_bias, B, N, H,
                               wait_base(status), stream, &tmap_ok);
  if (!tmap_ok) return EVOATTN_ERR_ALIGNMENT;
  return cuda_status(e);
}

evoattn_status evoattn_transition(const void* z, const void* o, const void* w_o,
                                  const float* gamma, const float* beta, const void* w1,
                                  const void* w2, float eps, void* out, int B, int N, int C,
                                  int HD, int F, cudaStream_t stream) {
  if (!z || !gamma || !beta || !w1 || !w2 || !out) return EVOATTN_ERR_INVALID_ARG;
  if ((o == nullptr) != (w_o == nullptr)) return EVOATTN_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || C < 1 || F < 1 || (o && HD < 1)) return EVOATTN_ERR_INVALID_ARG;
  if (!(eps > 0.f) || !(eps < INFINITY)) return EVOATTN_ERR_INVALID_ARG;
  if (C != 128 || F != 4 * C || (o && HD != 128)) return EVOATTN_ERR_UNSUPPORTED;
  if ((uint64_t)B * N * N + 128 > 0x7FFFFFFFull) return EVOATTN_ERR_UNSUPPORTED;
  auto a16 = [](const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; };
  if (!a16(z) || !a16(w1) || !a16(w2) || !a16(out) || !a16(o) || !a16(w_o) ||
      reinterpret_cast<uintptr_t>(gamma) % 4 || reinterpret_cast<uintptr_t>(beta) % 4)
    return EVOATTN_ERR_ALIGNMENT;
  bool ok = false;
  unsigned int* status = status_word(&ok);
  if (!ok) return EVOATTN_ERR_CUDA;
  bool tmap_ok = true;
  cudaError_t e = bf16_transition(z, o, w_o, gamma, beta, w1, w2, eps, out, B, N,
                                  wait_base(status), stream, &tmap_ok);
  if (!tmap_ok) return EVOATTN_ERR_ALIGNMENT;
  return cuda_status(e);
}

evoattn_status evoattn_get_device_status(cudaStream_t stream, int* device_status) {
  if (!device_status) return EVOATTN_ERR_INVALID_ARG;
  bool ok = false;
  unsigned int* w = status_word(&ok);
  if (!ok) return EVOATTN_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return EVOATTN_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return EVOATTN_ERR_CUDA;
  if (v != 0 && cudaMemset(w, 0, sizeof(v)) != cudaSuccess) return EVOATTN_ERR_CUDA;  // word [0] only
  *device_status = (v & (1u << EVOATTN_ERR_TIMEOUT)) ? EVOATTN_ERR_TIMEOUT : EVOATTN_OK;
  return EVOATTN_OK;
}

evoattn_status evoattn_fwd(const void* q, const int64_t q_strides[5], const void* k,
                           const int64_t k_strides[5], const void* v,
                           const int64_t v_strides[5], const void* pair_bias,
                           const int64_t bias_strides[4], const uint8_t* mask,
                           const int64_t mask_strides[3], const void* gate,
                           const int64_t gate_strides[5], void* out,
                           const int64_t out_strides[5], float* lse, int B, int S, int H,
                           int N, int D, evoattn_dtype dtype, cudaStream_t stream) {
  if (!q || !k || !v || !pair_bias || !out || !lse) return EVOATTN_ERR_INVALID_ARG;
  if (!q_strides || !k_strides || !v_strides || !bias_strides || !out_strides)
    return EVOATTN_ERR_INVALID_ARG;
  if ((mask && !mask_strides) || (gate && !gate_strides)) return EVOATTN_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || H < 1 || N < 1 || D < 1) return EVOATTN_ERR_INVALID_ARG;
  if (dtype != EVOATTN_BF16 && dtype != EVOATTN_F32) return EVOATTN_ERR_UNSUPPORTED;
  if (!d_supported(dtype, D)) return EVOATTN_ERR_UNSUPPORTED;
  if (!nonneg(q_strides, 5) || !nonneg(k_strides, 5) || !nonneg(v_strides, 5) ||
      !nonneg(bias_strides, 4) || !nonneg(out_strides, 5) ||
      (mask && !nonneg(mask_strides, 3)) || (gate && !nonneg(gate_strides, 5)))
    return EVOATTN_ERR_INVALID_ARG;

  Problem P{};
  P.B = B; P.S = S; P.H = H; P.N = N; P.D = D;
  P.q = s5(q_strides); P.k = s5(k_strides); P.v = s5(v_strides); P.o = s5(out_strides);
  if (gate) P.g = s5(gate_strides);
  P.bias = StridesBias{bias_strides[0], bias_strides[1], bias_strides[2], bias_strides[3]};
  if (mask) P.mask = StridesMask{mask_strides[0], mask_strides[1], mask_strides[2]};

  if (dtype == EVOATTN_BF16 &&
      (!bf16_ok5(q, q_strides) || !bf16_ok5(k, k_strides) || !bf16_ok5(v, v_strides) ||
       !bf16_ok5(out, out_strides) || (gate && !bf16_ok5(gate, gate_strides)) ||
       !bf16_ok_bias(pair_bias, bias_strides) || reinterpret_cast<uintptr_t>(lse) % 16))
    return EVOATTN_ERR_ALIGNMENT;

  bool ok = false;
  unsigned int* status = status_word(&ok);
  if (!ok) return EVOATTN_ERR_CUDA;

  if (dtype == EVOATTN_F32) {
    F32Ptrs a{};
    a.q = static_cast<const float*>(q); a.k = static_cast<const float*>(k);
    a.v = static_cast<const float*>(v); a.bias = static_cast<const float*>(pair_bias);
    a.gate = static_cast<const float*>(gate); a.mask = mask;
    a.out = static_cast<float*>(out); a.lse = lse;
    return cuda_status(f32_fwd(P, a, stream));
  }
  Bf16Ptrs a{};
  a.q = q; a.k = k; a.v = v; a.bias = pair_bias; a.gate = gate; a.mask = mask;
  a.out = out; a.lse = lse;
  bool tmap_ok = true;
  cudaError_t e = bf16_fwd(P, a, wait_base(status), stream, &tmap_ok);
  if (!tmap_ok) return EVOATTN_ERR_ALIGNMENT;
  return cuda_status(e);
}

size_t evoattn_bwd_workspace_size(int B, int S, int H, int N, int D, evoattn_dtype dtype,
                                  unsigned flags) {
  if (B < 1 || S < 1 || H < 1 || N < 1 || !d_supported_bwd(dtype, D) || (flags & ~7u)) return 0;
  Problem P{};
  P.B = B; P.S = S; P.H = H; P.N = N; P.D = D;
  return dtype == EVOATTN_F32 ? f32_bwd_workspace_bytes(P) : bf16_bwd_workspace_bytes(P, flags);
}

static evoattn_status bwd_impl(const void* q, const int64_t q_strides[5], const void* k,
                           const int64_t k_strides[5], const void* v,
                           const int64_t v_strides[5], const void* pair_bias,
                           const int64_t bias_strides[4], const uint8_t* mask,
                           const int64_t mask_strides[3], const void* gate,
                           const int64_t gate_strides[5], const void* out,
                           const int64_t out_strides[5], const float* lse, const void* dout,
                           const int64_t dout_strides[5], void* dq,
                           const int64_t dq_strides[5], void* dk,
                           const int64_t dk_strides[5], void* dv,
                           const int64_t dv_strides[5], float* dbias, void* dgate,
                           const int64_t dgate_strides[5], int B, int S, int H, int N, int D,
                           evoattn_dtype dtype, unsigned flags, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream, cudaEvent_t* events) {
  if (!q || !k || !v || !pair_bias || !out || !lse || !dout || !dq || !dk || !dv || !dbias)
    return EVOATTN_ERR_INVALID_ARG;
  if (!q_strides || !k_strides || !v_strides || !bias_strides || !out_strides ||
      !dout_strides || !dq_strides || !dk_strides || !dv_strides)
    return EVOATTN_ERR_INVALID_ARG;
  if ((mask && !mask_strides) || (gate && !gate_strides)) return EVOATTN_ERR_INVALID_ARG;
  if ((gate == nullptr) != (dgate == nullptr)) return EVOATTN_ERR_INVALID_ARG;
  if (dgate && !dgate_strides) return EVOATTN_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || H < 1 || N < 1 || D < 1) return EVOATTN_ERR_INVALID_ARG;
  if (flags & ~7u) return EVOATTN_ERR_INVALID_ARG;
  if (dtype != EVOATTN_BF16 && dtype != EVOATTN_F32) return EVOATTN_ERR_UNSUPPORTED;
  if (!d_supported_bwd(dtype, D)) return EVOATTN_ERR_UNSUPPORTED;
  if (!nonneg(q_strides, 5) || !nonneg(k_strides, 5) || !nonneg(v_strides, 5) ||
      !nonneg(bias_strides, 4) || !nonneg(out_strides, 5) || !nonneg(dout_strides, 5) ||
      !nonneg(dq_strides, 5) || !nonneg(dk_strides, 5) || !nonneg(dv_strides, 5) ||
      (mask && !nonneg(mask_strides, 3)) || (gate && !nonneg(gate_strides, 5)) ||
      (dgate && !nonneg(dgate_strides, 5)))
    return EVOATTN_ERR_INVALID_ARG;
  const size_t need = evoattn_bwd_workspace_size(B, S, H, N, D, dtype, flags);
  if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256)
    return EVOATTN_ERR_WORKSPACE;

  Problem P{};
  P.B = B; P.S = S; P.H = H; P.N = N; P.D = D;
  P.q = s5(q_strides); P.k = s5(k_strides); P.v = s5(v_strides); P.o = s5(out_strides);
  P.dout = s5(dout_strides); P.dq = s5(dq_strides); P.dk = s5(dk_strides);
  P.dv = s5(dv_strides);
  if (gate) { P.g = s5(gate_strides); P.dg = s5(dgate_strides); }
  P.bias = StridesBias{bias_strides[0], bias_strides[1], bias_strides[2], bias_strides[3]};
  if (mask) P.mask = StridesMask{mask_strides[0], mask_strides[1], mask_strides[2]};

  if (dtype == EVOATTN_BF16 &&
      (!bf16_ok5(q, q_strides) || !bf16_ok5(k, k_strides) || !bf16_ok5(v, v_strides) ||
       !bf16_ok5(out, out_strides) || !bf16_ok5(dout, dout_strides) ||
       !bf16_ok5(dq, dq_strides) || !bf16_ok5(dk, dk_strides) || !bf16_ok5(dv, dv_strides) ||
       (gate && (!bf16_ok5(gate, gate_strides) || !bf16_ok5(dgate, dgate_strides))) ||
       !bf16_ok_bias(pair_bias, bias_strides) || reinterpret_cast<uintptr_t>(lse) % 16 ||
       reinterpret_cast<uintptr_t>(dbias) % 16))
    return EVOATTN_ERR_ALIGNMENT;

  bool ok = false;
  unsigned int* status = status_word(&ok);
  if (!ok) return EVOATTN_ERR_CUDA;

  if (dtype == EVOATTN_F32) {
    F32Ptrs a{};
    a.q = static_cast<const float*>(q); a.k = static_cast<const float*>(k);
    a.v = static_cast<const float*>(v); a.bias = static_cast<const float*>(pair_bias);
    a.gate = static_cast<const float*>(gate); a.mask = mask;
    a.dout = static_cast<const float*>(dout);
    a.out = const_cast<float*>(static_cast<const float*>(out));
    a.lse = const_cast<float*>(lse);
    a.dq = static_cast<float*>(dq); a.dk = static_cast<float*>(dk);
    a.dv = static_cast<float*>(dv); a.dbias = dbias; a.dgate = static_cast<float*>(dgate);
    return cuda_status(f32_bwd(P, a, workspace, stream, events));
  }
  Bf16Ptrs a{};
  a.q = q; a.k = k; a.v = v; a.bias = pair_bias; a.gate = gate; a.mask = mask;
  a.dout = dout; a.out = const_cast<void*>(out); a.lse = const_cast<float*>(lse);
  a.dq = dq; a.dk = dk; a.dv = dv; a.dgate = dgate; a.dbias = dbias;
  bool tmap_ok = true;
  cudaError_t e = bf16_bwd(P, a, flags, workspace, wait_base(status), stream, &tmap_ok, events);
  if (!tmap_ok) return EVOATTN_ERR_ALIGNMENT;
  return cuda_status(e);
}

evoattn_status evoattn_bwd(const void* q, const int64_t q_strides[5], const void* k,
                           const int64_t k_strides[5], const void* v,
                           const int64_t v_strides[5], const void* pair_bias,
                           const int64_t bias_strides[4], const uint8_t* mask,
                           const int64_t mask_strides[3], const void* gate,
                           const int64_t gate_strides[5], const void* out,
                           const int64_t out_strides[5], const float* lse, const void* dout,
                           const int64_t dout_strides[5], void* dq,
                           const int64_t dq_strides[5], void* dk,
                           const int64_t dk_strides[5], void* dv,
                           const int64_t dv_strides[5], float* dbias, void* dgate,
                           const int64_t dgate_strides[5], int B, int S, int H, int N, int D,
                           evoattn_dtype dtype, unsigned flags, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  return bwd_impl(q, q_strides, k, k_strides, v, v_strides, pair_bias, bias_strides, mask,
                  mask_strides, gate, gate_strides, out, out_strides, lse, dout, dout_strides,
                  dq, dq_strides, dk, dk_strides, dv, dv_strides, dbias, dgate, dgate_strides,
                  B, S, H, N, D, dtype, flags, workspace, workspace_bytes, stream, nullptr);
}

evoattn_status evoattn_bwd_profiled(const void* q, const int64_t q_strides[5], const void* k,
                                    const int64_t k_strides[5], const void* v,
                                    const int64_t v_strides[5], const void* pair_bias,
                                    const int64_t bias_strides[4], const uint8_t* mask,
                                    const int64_t mask_strides[3], const void* gate,
                                    const int64_t gate_strides[5], const void* out,
                                    const int64_t out_strides[5], const float* lse,
                                    const void* dout, const int64_t dout_strides[5], void* dq,
                                    const int64_t dq_strides[5], void* dk,
                                    const int64_t dk_strides[5], void* dv,
                                    const int64_t dv_strides[5], float* dbias, void* dgate,
                                    const int64_t dgate_strides[5], int B, int S, int H, int N,
                                    int D, evoattn_dtype dtype, unsigned flags,
                                    void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream, cudaEvent_t stage_events[5]) {
  if (!stage_events) return EVOATTN_ERR_INVALID_ARG;
  return bwd_impl(q, q_strides, k, k_strides, v, v_strides, pair_bias, bias_strides, mask,
                  mask_strides, gate, gate_strides, out, out_strides, lse, dout, dout_strides,
                  dq, dq_strides, dk, dk_strides, dv, dv_strides, dbias, dgate, dgate_strides,
                  B, S, H, N, D, dtype, flags, workspace, workspace_bytes, stream, stage_events);
}

}  // extern "C"
