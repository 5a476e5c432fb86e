// Internal interface between the C-ABI layer (m3_api.cu) and the kernels.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "m3_ssm.h"

namespace m3 {

// Validated arguments of one prefill call.  State pointers are null when the
// caller passed no entry state (fresh sequence) or wants no exit state.
struct PrefillArgs {
  m3_dims d;
  const void* x;
  const void* B;
  const void* C;
  const void* dt;
  const float* A;
  const void* lam;
  const void* theta;
  m3_state h0;  // all members null for a fresh sequence
  void* y;
  m3_state hT;  // all members null when no exit state is wanted
  unsigned* status;  // device status word (first bytes of the workspace)
  uint8_t* ws;       // the workspace (status word first)
  const m3_bc_norm* norm;  // BCNorm + biases applied to B and C on the fly, or null
};

struct DecodeArgs {
  m3_dims d;
  m3_state s;
  const void* x;
  const void* B;
  const void* C;
  const void* dt;
  const float* A;
  const void* lam;
  const void* theta;
  void* y;
  const m3_bc_norm* norm;  // BCNorm + biases applied to B_t, C_t and prev_B, or null
};

// Tensor-core (tcgen05) chunked prefill: bf16 inputs, P = 64, N in {64, 128}, R in {1,2,4,8}.
bool prefill_tc_supported(const m3_dims& d);

// How the tensor-core prefill splits long sequences, and where the per-segment arrays sit
// in the workspace (byte offsets; bytes = total workspace, status word included).
struct TcSegments {
  int nseg, seg_len;
  size_t off_u, off_h, off_d, off_dphi, off_phi, bytes;
};
TcSegments tc_segments(const m3_dims& d);
int sm_count();
cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s);

// CUDA-core recurrent prefill (fp32 arithmetic): every shape the API accepts.
bool prefill_recurrent_supported(const m3_dims& d);
cudaError_t launch_prefill_recurrent(const PrefillArgs& a, cudaStream_t s);

bool decode_supported(const m3_dims& d);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);

// Backward pass of the prefill (CUDA cores, fp32; the chunked masked form transposed).
struct BackwardArgs {
  m3_dims d;
  const void* x;
  const void* B;
  const void* C;
  const void* dt;
  const float* A;
  const void* lam;
  const void* theta;
  m3_state h0;  // all members null for a fresh sequence
  const void* dy;
  const float* dhT;  // null: no gradient on the exit state
  float* dx;
  float* dB;
  float* dC;
  float* ddt;
  float* dA;
  float* dlam;
  float* dtheta;
  float* dh0;  // null: not wanted
  uint8_t* ws;
};
struct BackwardWorkspace {
  int c, nch;  // tokens per chunk, chunks per sequence
  size_t off_da, off_da_chunk, off_dec, off_dqf, off_sig, off_sphi, off_dh0, off_h, off_g, bytes;
};
BackwardWorkspace backward_workspace(const m3_dims& d);
bool backward_supported(const m3_dims& d);
cudaError_t launch_backward(const BackwardArgs& a, cudaStream_t s);

}  // namespace m3
