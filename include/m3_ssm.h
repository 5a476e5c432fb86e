/*
 * m3_ssm.h -- C ABI of the Mamba-3 SSM layer core on NVIDIA B300 (sm_103a).
 *
 * What the library computes (paper: "Mamba-3: Improved Sequence Modeling
 * using State Space Principles"):
 *
 *   For every batch row b and head h independently, over tokens t:
 *     alpha_t = exp(dt_t A_h),  beta_t = (1 - lambda_t) dt_t alpha_t,
 *     gamma_t = lambda_t dt_t                                   (Proposition 1)
 *     phi_t   = phi_{t-1} + dt_t theta_t   (one angle per state pair (2k, 2k+1))
 *     B~_t = R(phi_t)^T B_t,  C~_t = R(phi_t)^T C_t             (Proposition 3)
 *     h_t = alpha_t h_{t-1} + beta_t B~_{t-1} X_{t-1}^T + gamma_t B~_t X_t^T
 *                                      (Proposition 4; MIMO rank R, section 3.3)
 *     y_t = h_t^T C~_t                                          (P x R)
 *   with R(phi)^T (u, v) = (cos(phi) u + sin(phi) v, -sin(phi) u + cos(phi) v)
 *   and B~_{t-1} the previous token's B rotated by its own angle phi_{t-1}.
 *
 * Layouts: row-major, innermost index last, densely packed, no strides.
 *   x, y      [B][T][H][R][P]   (x[b,t,h,r,p] = X_t[p, r] of head h)
 *   B, C      [B][T][H][R][N]   (B[b,t,h,r,n] = B_t[n, r])
 *   dt,lambda [B][T][H]
 *   theta     [B][T][H][N/2]
 *   A         [H]                float32
 *   state:  h [B][H][N][P] float32;  phi [B][H][N/2] float32;
 *           prev_B [B][H][R][N], prev_x [B][H][R][P] in the input dtype
 *           (the raw, unrotated previous token; phi is its angle).
 * R = 1 is the SISO model; the R axis then has extent 1.
 *
 * Ownership: every pointer is device memory owned by the caller.  The
 * library allocates no device memory.  All calls are asynchronous on the
 * given stream (a cudaStream_t passed as void*; NULL = legacy default
 * stream).  Argument errors are found on the host before anything is
 * enqueued and are returned synchronously; nothing is launched then.
 * Launch failures return M3_ERR_CUDA.  Errors found on the device (a bounded
 * wait that ran out) are recorded in the workspace and read back with
 * m3_ssm_device_status.
 *
 * All pointers must be 16-byte aligned (M3_ERR_ALIGN otherwise).
 */
#ifndef M3_SSM_H_
#define M3_SSM_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  M3_OK = 0,
  M3_ERR_ARG = 1,         /* null pointer where one is required, bad enum value */
  M3_ERR_SHAPE = 2,       /* a size is negative, odd N, unsupported R, too large */
  M3_ERR_DTYPE = 3,       /* dtype combination not supported */
  M3_ERR_ALIGN = 4,       /* a pointer is not 16-byte aligned */
  M3_ERR_CUDA = 5,        /* a CUDA launch or call failed */
  M3_ERR_TIMEOUT = 6,     /* a device-side bounded wait ran out (see m3_ssm_device_status) */
  M3_ERR_UNSUPPORTED = 7, /* valid request this build does not implement */
  M3_ERR_WORKSPACE = 8,   /* workspace missing or smaller than m3_ssm_prefill_workspace() */
  M3_ERR_RANGE = 9        /* an input exceeded the tensor-core path's fp16 operand range
                             (see m3_ssm_prefill; reported by m3_ssm_device_status) */
} m3_status;

typedef enum { M3_F32 = 0, M3_BF16 = 1 } m3_dtype;

typedef struct {
  int B;              /* batch rows */
  int T;              /* tokens (prefill); ignored by the decode step */
  int H;              /* heads */
  int P;              /* head dimension (multiple of 4, <= 256) */
  int N;              /* state dimension (even, <= 256); N/2 rotation pairs */
  int R;              /* MIMO rank: 1, 2, 4 or 8 (1 = SISO) */
  int chunk;          /* prefill chunk length in tokens, a hint (>= 0; 0 = the
                         kernel's own choice).  The result does not depend on it:
                         the chunked form is the same linear map as the recurrence,
                         reassociated.  The bf16 tensor-core kernel always runs
                         chunks of 128 (token, rank) rows, i.e. 128/R tokens, and
                         the fp32 recurrent kernel runs token by token, whatever
                         value is passed. */
  m3_dtype in_dtype;  /* x, B, C, dt, lambda, theta, prev_B, prev_x */
  m3_dtype out_dtype; /* y */
} m3_dims;

typedef struct {
  float* h;     /* [B][H][N][P] */
  float* phi;   /* [B][H][N/2] */
  void* prev_B; /* [B][H][R][N], in_dtype */
  void* prev_x; /* [B][H][R][P], in_dtype */
} m3_state;

/*
 * Bytes of device workspace m3_ssm_prefill needs for these dimensions
 * (always >= 256).  The workspace must be zero-filled before its first use;
 * the library leaves it ready for the next call afterwards.  One workspace
 * may serve calls that are ordered on one stream, not calls that overlap.
 */
size_t m3_ssm_prefill_workspace(const m3_dims* dims);

/*
 * Chunked prefill over T tokens (paper section 2.3 and Eq. (7): the masked
 * matrix form, decay mask times the 2-band convolution matrix; chunked as in
 * section 3.3 "parallel within a chunk, recurrent across chunks").
 *
 *   h0   entry state, or NULL for a fresh sequence (h = 0, phi = 0, no previous
 *        token).  Read only.
 *   y    output [B][T][H][R][P] in out_dtype.
 *   hT   exit state (h_T, phi_T, prev_B = B_{T-1}, prev_x = x_{T-1}), or NULL.
 *        hT may alias h0 member by member (in-place continuation).  With
 *        T = 0, hT receives a copy of h0 (or the zero state).
 *   workspace / ws_bytes: caller-owned scratch, see m3_ssm_prefill_workspace.
 *
 * bf16 inputs with P = 64, N in {64, 128}, R in {1, 2, 4, 8} run on the
 * tcgen05 tensor-core kernel; every other supported shape, and fp32 inputs,
 * run on a CUDA-core recurrent kernel with fp32 arithmetic.
 *
 * Tensor-core operands: the rotated B and C and the products dt-weight * x are
 * held as fp16 (the state copy is rescaled per chunk, the masked scores are
 * bf16 hi + lo pairs), with fp32 accumulation; the result is within about 1% of
 * the output RMS of the exact recurrence.  An operand value beyond the fp16
 * range (|B|, |C| above about 46000, or |x| times the step weight above 65504)
 * makes m3_ssm_device_status report M3_ERR_RANGE for that call; its outputs
 * are then invalid.
 */
m3_status m3_ssm_prefill(const m3_dims* dims, const void* x, const void* B, const void* C,
                         const void* dt, const float* A, const void* lambda, const void* theta,
                         const m3_state* h0, void* y, const m3_state* hT, void* workspace,
                         size_t ws_bytes, void* stream);

/*
 * One decode step (the recurrence above for a single token; paper section
 * 3.3 and Table 6's single-token decode).  `state` is read and updated in
 * place: h <- h', phi <- phi + dt theta, prev_B <- B_t, prev_x <- x_t.
 * Per-token inputs have the prefill layouts with T = 1:
 *   x_t [B][H][R][P], B_t/C_t [B][H][R][N], dt_t/lambda_t [B][H], theta_t [B][H][N/2].
 *   y_t [B][H][R][P] in out_dtype.
 * dims->T and dims->chunk are ignored.  No workspace is used.
 */
m3_status m3_ssm_decode_step(const m3_dims* dims, const m3_state* state, const void* x_t,
                             const void* B_t, const void* C_t, const void* dt_t, const float* A,
                             const void* lambda_t, const void* theta_t, void* y_t, void* stream);

/*
 * Waits for `stream`, then reads and clears the device status word kept in
 * `workspace`.  Returns M3_OK, M3_ERR_TIMEOUT (a bounded wait inside a
 * prefill kernel ran out; that call's outputs are invalid), M3_ERR_RANGE (an
 * operand exceeded the tensor-core path's fp16 range; outputs invalid), or
 * M3_ERR_CUDA.
 */
m3_status m3_ssm_device_status(void* workspace, void* stream);

/*
 * m3_ssm_prefill for callers that cannot allocate device memory.  The paper has
 * no counterpart to this call; it exists for hosts that forbid device allocation
 * once they are running (cudaMalloc synchronises the device and can fail under
 * memory pressure), such as plugin hosts and serving loops, and for code whose
 * whole memory budget belongs to a pool it does not control.
 *
 * Same arguments, layouts and results as m3_ssm_prefill, without the workspace:
 * the scratch comes from a 4 MiB array in the library's device image, which
 * every GPU that loads the library holds until the process exits.  The call
 * allocates nothing (no cudaMalloc, no cudaFree, no allocating library routine).
 *   - The first call on a device looks up the array's device address on the
 *     current device (cudaGetSymbolAddress) and caches it; make that first call
 *     before any stream capture on that device.  The scratch used is that of the
 *     device current at the call, which must be the device holding the tensors.
 *     cudaDeviceReset invalidates the cached address: do not call this entry point
 *     on a device after resetting it in the same process.
 *   - Each call clears the part of the array it uses (cudaMemsetAsync on
 *     `stream`) before the kernels run.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind: calls whose work overlaps on the GPU (different streams, no
 *     ordering between them) race on it.  Order such calls on one stream.
 *   - Returns M3_ERR_WORKSPACE if m3_ssm_prefill_workspace(dims) exceeds
 *     4 MiB, M3_ERR_CUDA if the address lookup or the clear fails, and
 *     otherwise whatever m3_ssm_prefill returns for the same arguments.
 *   - A device-side wait that ran out is recorded in the array's status word,
 *     which the caller cannot reach; it is cleared by the next call.  Callers
 *     that need that report use m3_ssm_prefill with their own workspace.
 */
m3_status m3_ssm_prefill_noalloc(const m3_dims* dims, const void* x, const void* B, const void* C,
                                 const void* dt, const float* A, const void* lambda,
                                 const void* theta, const m3_state* h0, void* y,
                                 const m3_state* hT, void* stream);

/*
 * BCNorm and the B, C biases fused into the SSM core (paper section 3.4, "BC / QK
 * normalisation": an RMS normalisation right after the B and C projections, in the manner
 * of QKNorm; "B, C bias": a learnable, head-specific, channel-wise bias added after the
 * normalisation).  The pages give no formula; this library reads it as
 *
 *   B_t[:, r] = Braw_t[:, r] / sqrt(mean_n Braw_t[n, r]^2 + eps) * B_weight + B_bias[h]
 *
 * per (token, head, rank) vector of N state entries, likewise for C with its own weight and
 * bias, and the result feeds the recurrence above in place of B and C.
 *
 *   B_weight, C_weight  [N] in the input dtype, shared by heads and ranks; NULL = all ones.
 *   B_bias,   C_bias    [H][N] in the input dtype, shared by ranks; NULL = all zeros.
 *   eps                 > 0 (and finite), added to the mean square.
 */
typedef struct {
  const void* B_weight;
  const void* B_bias;
  const void* C_weight;
  const void* C_bias;
  float eps;
} m3_bc_norm;

/*
 * m3_ssm_prefill on the raw projection outputs: B and C are the [B][T][H][R][N] values
 * before BCNorm and the biases, which the kernels apply on the fly (the normalised B and C
 * never go through device memory).  The state keeps the raw previous token: h0->prev_B and
 * hT->prev_B hold the raw B of the last token, normalised again with `norm` when its
 * trapezoid term is folded in, so continuation calls must pass the same `norm`.
 * Every other argument, the workspace (sized by m3_ssm_prefill_workspace for the same dims),
 * the supported shapes and the error behaviour are those of m3_ssm_prefill; `norm` must not
 * be NULL (M3_ERR_ARG), eps must be > 0 and finite (M3_ERR_ARG), and the four parameter
 * pointers must be 16-byte aligned or NULL (M3_ERR_ALIGN).
 */
m3_status m3_ssm_prefill_bcnorm(const m3_dims* dims, const void* x, const void* B_raw,
                                const void* C_raw, const void* dt, const float* A,
                                const void* lambda, const void* theta, const m3_bc_norm* norm,
                                const m3_state* h0, void* y, const m3_state* hT, void* workspace,
                                size_t ws_bytes, void* stream);

/*
 * m3_ssm_decode_step on the raw projection outputs B_t, C_t [B][H][R][N], with BCNorm and
 * the biases applied in the step's prologue.  state->prev_B holds the raw previous B (see
 * m3_ssm_prefill_bcnorm) and receives the raw B_t.  Arguments and errors as
 * m3_ssm_decode_step, and `norm` as m3_ssm_prefill_bcnorm.
 */
m3_status m3_ssm_decode_step_bcnorm(const m3_dims* dims, const m3_state* state, const void* x_t,
                                    const void* B_raw_t, const void* C_raw_t, const void* dt_t,
                                    const float* A, const void* lambda_t, const void* theta_t,
                                    const m3_bc_norm* norm, void* y_t, void* stream);

/*
 * The Mamba-2 special case of the same layer core (paper section 2, Eq. (4), the
 * exponential-Euler rule that Mamba-1 and Mamba-2 use, and Remark 5: the mask keeps
 * only its diagonal weights), for the Mamba-2 versus Mamba-3 comparison of Table 6:
 *
 *   h_t = exp(dt_t A_h) h_{t-1} + dt_t B_t X_t^T,   y_t = h_t^T C_t
 *
 * i.e. the recurrence above with lambda = 1 (no trapezoid term) and theta = 0 (a real
 * transition, no rotation).  SISO only (dims->R must be 1).  The state is h alone:
 *   h0, hT, h   [B][H][N][P] float32 device pointers; h0 may be NULL (zero state), hT
 *               may be NULL (not written) or equal h0 (in-place continuation).
 * x, B, C, dt, A, y and their layouts, dtypes, alignment, workspace (sized by
 * m3_ssm_prefill_workspace for the same dims), stream and status behaviour are those of
 * m3_ssm_prefill / m3_ssm_decode_step.  The bf16 prefill with P = 64, N in {64, 128} runs
 * on the tensor-core kernel with the rotation and the lambda terms compiled out; the
 * decode step reads and writes the state exactly once.
 */
m3_status m3_ssd_prefill(const m3_dims* dims, const void* x, const void* B, const void* C,
                         const void* dt, const float* A, const float* h0, void* y, float* hT,
                         void* workspace, size_t ws_bytes, void* stream);

m3_status m3_ssd_decode_step(const m3_dims* dims, float* h, const void* x_t, const void* B_t,
                             const void* C_t, const void* dt_t, const float* A, void* y_t,
                             void* stream);

/*
 * Backward pass of m3_ssm_prefill: the gradients a training step needs (paper section 1,
 * "fast training kernels"; the masked form of section 2.3 / Eq. (7) is the same linear map
 * as the recurrence, whose adjoint is run in reverse time).  For the loss
 * L = <dy, y> + <dhT, h_T> of one prefill call with the given inputs and entry state:
 *
 *   dy     cotangent of y, [B][T][H][R][P] in dims->out_dtype (the dtype y had).
 *   dhT    cotangent of the exit state h_T, float [B][H][N][P], or NULL (zero).
 *   h0     the entry state the forward call used, or NULL (fresh sequence).
 *   dx     float [B][T][H][R][P];   dB, dC float [B][T][H][R][N];
 *   ddt, dlambda  float [B][T][H];  dtheta float [B][T][H][N/2];
 *   dA     float [H], summed over batch rows and tokens (overwritten);
 *   dh0    float [B][H][N][P], gradient with respect to the entry state's h, or NULL.
 *          Gradients with respect to the entry state's angle and previous token are not
 *          produced.
 * All gradients are fp32 whatever the input dtype; the arithmetic is fp32 on CUDA cores in
 * the chunked masked form, with chunks of up to 32 tokens (at most 64 (token, rank) rows):
 * every chunk's own contributions to the states around it, in parallel over all chunks; a
 * scan from chunk to chunk of the chunk-entry states and of the exit-state cotangents (fp32
 * in the workspace, 2 N P floats per chunk); then every chunk's adjoint, in parallel.  Every
 * reduction has a fixed order: results are bit-identical from run to run.  Supported when
 * N * P <= 8192, N even and N <= 1024; other shapes return M3_ERR_SHAPE.  Inputs, dtypes,
 * alignment and stream behaviour as m3_ssm_prefill; the workspace must hold
 * m3_ssm_prefill_backward_workspace bytes (its contents need no initialisation); a bounded
 * wait inside the kernels that ran out is recorded in the workspace's status word, read with
 * m3_ssm_device_status(workspace) after the call (M3_ERR_TIMEOUT).  dims->chunk is ignored.
 */
size_t m3_ssm_prefill_backward_workspace(const m3_dims* dims);

m3_status m3_ssm_prefill_backward(const m3_dims* dims, const void* x, const void* B, const void* C,
                                  const void* dt, const float* A, const void* lambda,
                                  const void* theta, const m3_state* h0, const void* dy,
                                  const float* dhT, float* dx, float* dB, float* dC, float* ddt,
                                  float* dA, float* dlambda, float* dtheta, float* dh0,
                                  void* workspace, size_t ws_bytes, void* stream);

/* Short English description of a status code (static storage). */
const char* m3_status_str(m3_status s);

#ifdef __cplusplus
}
#endif

#endif /* M3_SSM_H_ */
