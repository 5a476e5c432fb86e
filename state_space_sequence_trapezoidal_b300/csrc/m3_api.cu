// C ABI of the Mamba-3 SSM core: argument validation on the host, dispatch to
// the kernels, status codes.  Nothing here allocates device memory.
#include <cuda_runtime.h>
#include <stdint.h>

#include "m3_internal.h"
#include "m3_ptx.cuh"

namespace {

constexpr size_t kStatusBytes = 256;  // status word + reserved, at the workspace start

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

m3_status check_dims(const m3_dims* d, bool prefill) {
  if (!d) return M3_ERR_ARG;
  if (d->in_dtype != M3_F32 && d->in_dtype != M3_BF16) return M3_ERR_DTYPE;
  if (d->out_dtype != M3_F32 && d->out_dtype != M3_BF16) return M3_ERR_DTYPE;
  if (d->B < 0 || d->H < 0 || (prefill && d->T < 0)) return M3_ERR_SHAPE;
  if (d->N < 2 || d->N > 256 || (d->N & 1)) return M3_ERR_SHAPE;
  if (d->P < 4 || d->P > 256 || (d->P & 3)) return M3_ERR_SHAPE;
  if (d->R != 1 && d->R != 2 && d->R != 4 && d->R != 8) return M3_ERR_SHAPE;
  if (prefill && d->chunk < 0) return M3_ERR_SHAPE;
  // element counts must fit the kernels' 32-bit grid and 64-bit offsets comfortably
  const long long bh = static_cast<long long>(d->B) * d->H;
  if (bh > 0x7fffffffLL) return M3_ERR_SHAPE;
  return M3_OK;
}

bool state_all_or_none(const m3_state* s) {
  const bool any = s->h || s->phi || s->prev_B || s->prev_x;
  const bool all = s->h && s->phi && s->prev_B && s->prev_x;
  return !any || all;
}

bool state_aligned(const m3_state* s) {
  return aligned16(s->h) && aligned16(s->phi) && aligned16(s->prev_B) && aligned16(s->prev_x);
}

// BCNorm parameters: eps > 0 and finite; parameter pointers 16-byte aligned or null.
m3_status check_norm(const m3_bc_norm* n) {
  if (!n) return M3_ERR_ARG;
  if (!(n->eps > 0.f) || !(n->eps < 3.0e38f)) return M3_ERR_ARG;
  if (!aligned16(n->B_weight) || !aligned16(n->B_bias) || !aligned16(n->C_weight) ||
      !aligned16(n->C_bias))
    return M3_ERR_ALIGN;
  return M3_OK;
}

}  // namespace

extern "C" {

size_t m3_ssm_prefill_workspace(const m3_dims* dims) {
  if (!dims || check_dims(dims, true) != M3_OK || !m3::prefill_tc_supported(*dims) || dims->T <= 0)
    return kStatusBytes;
  const size_t b = m3::tc_segments(*dims).bytes;
  return b > kStatusBytes ? b : kStatusBytes;
}

const char* m3_status_str(m3_status s) {
  switch (s) {
    case M3_OK: return "ok";
    case M3_ERR_ARG: return "invalid argument (null pointer or bad enum)";
    case M3_ERR_SHAPE: return "unsupported or invalid shape";
    case M3_ERR_DTYPE: return "unsupported dtype";
    case M3_ERR_ALIGN: return "pointer not 16-byte aligned";
    case M3_ERR_CUDA: return "CUDA error";
    case M3_ERR_TIMEOUT: return "device-side wait timed out";
    case M3_ERR_UNSUPPORTED: return "request not supported by this build";
    case M3_ERR_WORKSPACE: return "workspace missing or too small";
    case M3_ERR_RANGE: return "operand outside the tensor-core path's fp16 range";
  }
  return "unknown status";
}

}  // extern "C"

namespace {

// Shared by m3_ssm_prefill and m3_ssd_prefill; `ssd` selects the Mamba-2 special case
// (lambda and theta null, state h only).
m3_status prefill_common(const m3_dims* dims, const void* x, const void* B, const void* C,
                         const void* dt, const float* A, const void* lambda, const void* theta,
                         const m3_state* h0, void* y, const m3_state* hT, void* workspace,
                         size_t ws_bytes, void* stream, bool ssd, const m3_bc_norm* norm = nullptr,
                         bool with_norm = false) {
  m3_status st = check_dims(dims, true);
  if (st != M3_OK) return st;
  if (with_norm && (st = check_norm(norm)) != M3_OK) return st;
  const m3_dims& d = *dims;
  if (ssd && d.R != 1) return M3_ERR_SHAPE;
  if (!ssd && h0 && !state_all_or_none(h0)) return M3_ERR_ARG;
  if (!ssd && hT && !state_all_or_none(hT)) return M3_ERR_ARG;
  if (!workspace) return M3_ERR_WORKSPACE;
  if (ws_bytes < m3_ssm_prefill_workspace(dims)) return M3_ERR_WORKSPACE;
  const bool empty = d.B == 0 || d.H == 0;
  const bool has_tokens = !empty && d.T > 0;
  if (has_tokens && (!x || !B || !C || !dt || !y)) return M3_ERR_ARG;
  if (has_tokens && !ssd && (!lambda || !theta)) return M3_ERR_ARG;
  if (!empty && !A) return M3_ERR_ARG;
  if (!aligned16(x) || !aligned16(B) || !aligned16(C) || !aligned16(dt) || !aligned16(A) ||
      !aligned16(lambda) || !aligned16(theta) || !aligned16(y) || !aligned16(workspace))
    return M3_ERR_ALIGN;
  if ((h0 && !state_aligned(h0)) || (hT && !state_aligned(hT))) return M3_ERR_ALIGN;

  m3::PrefillArgs a{};
  a.d = d;
  a.x = x;
  a.B = B;
  a.C = C;
  a.dt = dt;
  a.A = A;
  a.lam = lambda;
  a.theta = theta;
  if (h0) a.h0 = *h0;
  a.y = y;
  if (hT) a.hT = *hT;
  a.status = static_cast<unsigned*>(workspace);
  a.ws = static_cast<uint8_t*>(workspace);
  if (!a.h0.h) a.h0 = m3_state{nullptr, nullptr, nullptr, nullptr};
  if (!a.hT.h) a.hT = m3_state{nullptr, nullptr, nullptr, nullptr};
  a.norm = with_norm ? norm : nullptr;

  // With no tokens the call only copies the entry state to the exit state.
  const bool tc = m3::prefill_tc_supported(d) && d.T > 0;
  if (!tc && !m3::prefill_recurrent_supported(d)) return M3_ERR_SHAPE;
  if (empty) return M3_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = tc ? m3::launch_prefill_tc(a, s) : m3::launch_prefill_recurrent(a, s);
  return e == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

}  // namespace

namespace {

m3_status decode_common(const m3_dims* dims, const m3_state* state, const void* x_t,
                        const void* B_t, const void* C_t, const void* dt_t, const float* A,
                        const void* lambda_t, const void* theta_t, void* y_t, void* stream,
                        const m3_bc_norm* norm, bool with_norm) {
  m3_status st = check_dims(dims, false);
  if (st != M3_OK) return st;
  if (with_norm && (st = check_norm(norm)) != M3_OK) return st;
  const m3_dims& d = *dims;
  if (!state) return M3_ERR_ARG;
  if (!m3::decode_supported(d)) return M3_ERR_SHAPE;
  if (d.B == 0 || d.H == 0) return M3_OK;
  if (!state->h || !state->phi || !state->prev_B || !state->prev_x || !x_t || !B_t || !C_t ||
      !dt_t || !A || !lambda_t || !theta_t || !y_t)
    return M3_ERR_ARG;
  if (!state_aligned(state) || !aligned16(x_t) || !aligned16(B_t) || !aligned16(C_t) ||
      !aligned16(dt_t) || !aligned16(A) || !aligned16(lambda_t) || !aligned16(theta_t) ||
      !aligned16(y_t))
    return M3_ERR_ALIGN;
  m3::DecodeArgs a{d, *state, x_t, B_t, C_t, dt_t, A, lambda_t, theta_t, y_t,
                   with_norm ? norm : nullptr};
  const cudaError_t e = m3::launch_decode(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

}  // namespace

extern "C" {

m3_status m3_ssm_prefill(const m3_dims* dims, const void* x, const void* B, const void* C,
                         const void* dt, const float* A, const void* lambda, const void* theta,
                         const m3_state* h0, void* y, const m3_state* hT, void* workspace,
                         size_t ws_bytes, void* stream) {
  return prefill_common(dims, x, B, C, dt, A, lambda, theta, h0, y, hT, workspace, ws_bytes,
                        stream, false);
}

m3_status m3_ssm_prefill_bcnorm(const m3_dims* dims, const void* x, const void* B_raw,
                                const void* C_raw, const void* dt, const float* A,
                                const void* lambda, const void* theta, const m3_bc_norm* norm,
                                const m3_state* h0, void* y, const m3_state* hT, void* workspace,
                                size_t ws_bytes, void* stream) {
  return prefill_common(dims, x, B_raw, C_raw, dt, A, lambda, theta, h0, y, hT, workspace,
                        ws_bytes, stream, false, norm, true);
}

m3_status m3_ssd_prefill(const m3_dims* dims, const void* x, const void* B, const void* C,
                         const void* dt, const float* A, const float* h0, void* y, float* hT,
                         void* workspace, size_t ws_bytes, void* stream) {
  const m3_state s0{const_cast<float*>(h0), nullptr, nullptr, nullptr};
  const m3_state s1{hT, nullptr, nullptr, nullptr};
  return prefill_common(dims, x, B, C, dt, A, nullptr, nullptr, h0 ? &s0 : nullptr, y,
                        hT ? &s1 : nullptr, workspace, ws_bytes, stream, true);
}


m3_status m3_ssm_decode_step(const m3_dims* dims, const m3_state* state, const void* x_t,
                             const void* B_t, const void* C_t, const void* dt_t, const float* A,
                             const void* lambda_t, const void* theta_t, void* y_t, void* stream) {
  return decode_common(dims, state, x_t, B_t, C_t, dt_t, A, lambda_t, theta_t, y_t, stream,
                       nullptr, false);
}

m3_status m3_ssm_decode_step_bcnorm(const m3_dims* dims, const m3_state* state, const void* x_t,
                                    const void* B_raw_t, const void* C_raw_t, const void* dt_t,
                                    const float* A, const void* lambda_t, const void* theta_t,
                                    const m3_bc_norm* norm, void* y_t, void* stream) {
  return decode_common(dims, state, x_t, B_raw_t, C_raw_t, dt_t, A, lambda_t, theta_t, y_t,
                       stream, norm, true);
}

size_t m3_ssm_prefill_backward_workspace(const m3_dims* dims) {
  if (!dims || check_dims(dims, true) != M3_OK || !m3::backward_supported(*dims)) return kStatusBytes;
  const size_t b = m3::backward_workspace(*dims).bytes;
  return b > kStatusBytes ? b : kStatusBytes;
}

m3_status m3_ssm_prefill_backward(const m3_dims* dims, const void* x, const void* B, const void* C,
                                  const void* dt, const float* A, const void* lambda,
                                  const void* theta, const m3_state* h0, const void* dy,
                                  const float* dhT, float* dx, float* dB, float* dC, float* ddt,
                                  float* dA, float* dlambda, float* dtheta, float* dh0,
                                  void* workspace, size_t ws_bytes, void* stream) {
  m3_status st = check_dims(dims, true);
  if (st != M3_OK) return st;
  const m3_dims& d = *dims;
  if (!m3::backward_supported(d)) return M3_ERR_SHAPE;
  if (h0 && !state_all_or_none(h0)) return M3_ERR_ARG;
  if (!workspace) return M3_ERR_WORKSPACE;
  if (ws_bytes < m3_ssm_prefill_backward_workspace(dims)) return M3_ERR_WORKSPACE;
  if (d.B == 0 || d.H == 0) return M3_OK;
  if (!A || !dA) return M3_ERR_ARG;
  if (d.T > 0 && (!x || !B || !C || !dt || !lambda || !theta || !dy || !dx || !dB || !dC || !ddt ||
                  !dlambda || !dtheta))
    return M3_ERR_ARG;
  if (!aligned16(x) || !aligned16(B) || !aligned16(C) || !aligned16(dt) || !aligned16(A) ||
      !aligned16(lambda) || !aligned16(theta) || !aligned16(dy) || !aligned16(dhT) ||
      !aligned16(dx) || !aligned16(dB) || !aligned16(dC) || !aligned16(ddt) || !aligned16(dA) ||
      !aligned16(dlambda) || !aligned16(dtheta) || !aligned16(dh0) || !aligned16(workspace))
    return M3_ERR_ALIGN;
  if (h0 && !state_aligned(h0)) return M3_ERR_ALIGN;
  m3::BackwardArgs a{};
  a.d = d;
  a.x = x;
  a.B = B;
  a.C = C;
  a.dt = dt;
  a.A = A;
  a.lam = lambda;
  a.theta = theta;
  a.h0 = (h0 && h0->h) ? *h0 : m3_state{nullptr, nullptr, nullptr, nullptr};
  a.dy = dy;
  a.dhT = dhT;
  a.dx = dx;
  a.dB = dB;
  a.dC = dC;
  a.ddt = ddt;
  a.dA = dA;
  a.dlam = dlambda;
  a.dtheta = dtheta;
  a.dh0 = dh0;
  a.ws = static_cast<uint8_t*>(workspace);
  const cudaError_t e = m3::launch_backward(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

m3_status m3_ssd_decode_step(const m3_dims* dims, float* h, const void* x_t, const void* B_t,
                             const void* C_t, const void* dt_t, const float* A, void* y_t,
                             void* stream) {
  m3_status st = check_dims(dims, false);
  if (st != M3_OK) return st;
  const m3_dims& d = *dims;
  if (d.R != 1 || !m3::decode_supported(d)) return M3_ERR_SHAPE;
  if (d.B == 0 || d.H == 0) return M3_OK;
  if (!h || !x_t || !B_t || !C_t || !dt_t || !A || !y_t) return M3_ERR_ARG;
  if (!aligned16(h) || !aligned16(x_t) || !aligned16(B_t) || !aligned16(C_t) || !aligned16(dt_t) ||
      !aligned16(A) || !aligned16(y_t))
    return M3_ERR_ALIGN;
  m3::DecodeArgs a{d, m3_state{h, nullptr, nullptr, nullptr}, x_t, B_t, C_t, dt_t, A, nullptr,
                   nullptr, y_t, nullptr};
  const cudaError_t e = m3::launch_decode(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

m3_status m3_ssm_device_status(void* workspace, void* stream) {
  if (!workspace) return M3_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return M3_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return M3_ERR_CUDA;
  if (word == 0) return M3_OK;
  if (cudaMemsetAsync(workspace, 0, sizeof(word), s) != cudaSuccess) return M3_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return M3_ERR_CUDA;
  if (word & m3::kDevTimeout) return M3_ERR_TIMEOUT;
  return (word & m3::kDevRange) ? M3_ERR_RANGE : M3_ERR_CUDA;
}

}  // extern "C"
