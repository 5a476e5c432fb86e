// Decode step of the Mamba-3 SSM core: one token, every (batch row, head).
//
// h' = alpha h + beta B~_{t-1} X_{t-1}^T + gamma B~_t X_t^T ; y = h'^T C~_t
// (Proposition 1 coefficients, Proposition 3 rotation, MIMO rank-R products
// of section 3.3).  The step is bound by the fp32 state stream: N x P x 4
// bytes read and written per (b, h), against O(N R + P R) bytes of per-token
// input.  One CTA owns one (b, h) slice; every thread issues all of its
// 16-byte state loads before the small prologue runs, so the state stream
// overlaps the rotation work.  The rank-R update and the output contraction
// read the rotated B~, C~ and X from shared memory; y is reduced over state
// rows in a fixed order (deterministic).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "m3_internal.h"

namespace m3 {
namespace {

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ void from_f(float& d, float v) { d = v; }
__device__ __forceinline__ void from_f(__nv_bfloat16& d, float v) { d = __float2bfloat16_rn(v); }

struct DecodeParams {
  float* h;
  float* phi;
  void* prevB;
  void* prevx;
  const void* x;
  const void* B;
  const void* C;
  const void* dt;
  const float* A;
  const void* lam;
  const void* theta;
  void* y;
  int H, N, P;
};

// BCNorm + biases (section 3.4) of B_t, C_t and the stored raw previous B, used when the
// kernel is built with kNorm: weights [N] (null: ones), biases [H][N] (null: zeros), in the
// input dtype.
struct DecodeNorm {
  const void* nwB;
  const void* nbB;
  const void* nwC;
  const void* nbC;
  float neps;
};

// 1 / RMS of each of the rows B_t[:, r], C_t[:, r], prev_B[:, r] (r < R) of this (b, h), into
// s_inv[3R]; a fixed summation order, so the result does not vary from run to run.  Whole
// warps each take one row; a block that is not a whole number of warps uses one thread per
// row.  Ends with a barrier.
template <typename Tin>
__device__ void row_inv_rms(const Tin* Bt, const Tin* Ct, const Tin* Bp, int R, int N, float eps,
                            float* s_inv) {
  if ((blockDim.x & 31) == 0) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    for (int j = warp; j < 3 * R; j += nwarps) {
      const Tin* row = (j < R ? Bt : j < 2 * R ? Ct : Bp) + static_cast<size_t>(j % R) * N;
      float ss = 0.f;
      for (int n = lane; n < N; n += 32) {
        const float v = to_f(row[n]);
        ss = fmaf(v, v, ss);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) s_inv[j] = rsqrtf(fmaf(ss, 1.f / N, eps));
    }
  } else {
    for (int j = threadIdx.x; j < 3 * R; j += blockDim.x) {
      const Tin* row = (j < R ? Bt : j < 2 * R ? Ct : Bp) + static_cast<size_t>(j % R) * N;
      float ss = 0.f;
      for (int n = 0; n < N; ++n) {
        const float v = to_f(row[n]);
        ss = fmaf(v, v, ss);
      }
      s_inv[j] = rsqrtf(fmaf(ss, 1.f / N, eps));
    }
  }
  __syncthreads();
}

// R consecutive floats of one state row (rank-major factors stored [N][R]).
template <int R>
__device__ __forceinline__ void load_r(const float* src, float (&v)[R]) {
  if constexpr (R % 4 == 0) {
#pragma unroll
    for (int q = 0; q < R / 4; ++q) {
      const float4 t = reinterpret_cast<const float4*>(src)[q];
      v[4 * q] = t.x;
      v[4 * q + 1] = t.y;
      v[4 * q + 2] = t.z;
      v[4 * q + 3] = t.w;
    }
  } else if constexpr (R == 2) {
    const float2 t = *reinterpret_cast<const float2*>(src);
    v[0] = t.x;
    v[1] = t.y;
  } else {
    v[0] = src[0];
  }
}

// Threads: (P/2) column pairs x RG row groups.  Thread (cg, rg) owns columns
// 2cg, 2cg+1 of rows rg, rg + RG, ..., rg + (VPT-1) RG.  The
// rotated factors sit in shared memory rank-innermost ([N][R]) and the token's
// X rows ([R][P]); each thread reads its own columns of X once and one short
// vector of factors per state row, so the update runs from registers.
// MAXT: 256 for the usual shapes, with enough CTAs per SM resident to keep the state
// stream in flight (the register budget shrinks with that count); 1024 for states too
// large to spread over 256 threads.
template <int R, int MAXT>
struct DecodeOcc {
  static constexpr int kMinBlocks = MAXT > 256 ? 1 : (R <= 4 ? 4 : 2);
};

// kRot = false: the Mamba-2 special case (lambda = 1, theta = 0, Eq. (4)): h' = alpha h +
// dt B_t X_t^T, y = h'^T C_t.  No angle, lambda or previous token is read or written.
// kNorm: B_t, C_t and the stored previous B are raw projection outputs; BCNorm (RMS over
// the N entries of each rank column, times a weight per state index) and the head's bias
// are applied before the rotation (section 3.4).
template <typename Tin, typename Tout, int R, int VPT, int MAXT, bool kRot, bool kNorm>
__global__ void __launch_bounds__(MAXT, DecodeOcc<R, MAXT>::kMinBlocks) decode_step_kernel(const DecodeParams p, const DecodeNorm q) {
  const int bh = blockIdx.x;
  const int head = bh % p.H;
  const int N = p.N, P = p.P, K = N >> 1;
  const int P2 = P >> 1;
  const int cg = threadIdx.x % P2;  // column pair
  const int rg = threadIdx.x / P2;
  const int RG = blockDim.x / P2;

  float* hs = p.h + static_cast<size_t>(bh) * N * P;
  float2 hv[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i)
    hv[i] = __ldcs(reinterpret_cast<const float2*>(hs + static_cast<size_t>(rg + i * RG) * P) + cg);

  extern __shared__ float sm[];
  float* sBt = sm;               // [N][R] B~_t
  float* sCt = sBt + R * N;      // [N][R] C~_t
  float* sBp = sCt + R * N;      // [N][R] B~_{t-1}
  float* sx = sBp + R * N;       // [R][P] X_t
  float* sxp = sx + R * P;       // [R][P] X_{t-1}
  float* red = sxp + R * P;      // [RG][R][P] partial outputs
  float* sphi = red + RG * R * P; // [K] advanced angle
  float* sinv = sphi + K;         // [3R] BCNorm 1/RMS of the B_t, C_t, prev_B columns

  const Tin* Bt = static_cast<const Tin*>(p.B);
  const Tin* Ct = static_cast<const Tin*>(p.C);
  Tin* prevB = static_cast<Tin*>(p.prevB);
  const float dt = to_f(static_cast<const Tin*>(p.dt)[bh]);
  const float lam = kRot ? to_f(static_cast<const Tin*>(p.lam)[bh]) : 1.f;
  const Tin* th = kRot ? static_cast<const Tin*>(p.theta) + static_cast<size_t>(bh) * K : nullptr;

  // Prologue, one round of loads: thread i < R K rotates column r, pair k of the previous
  // token (by its own angle phi) and of the current B and C (by phi + dt theta); thread
  // i < R P copies the token's x.  The advanced angle is stored back reduced to [-pi, pi]
  // so that long decode loops keep full precision.
  const Tin* xt = static_cast<const Tin*>(p.x) + static_cast<size_t>(bh) * R * P;
  Tin* prevx = kRot ? static_cast<Tin*>(p.prevx) + static_cast<size_t>(bh) * R * P : nullptr;
  if constexpr (!kRot) {
    for (int i = threadIdx.x; i < R * N || i < R * P; i += blockDim.x) {
      if (i < R * N) {  // element n of column r, stored [N][R]
        const int r = i / N, n = i - r * N;
        const size_t o = (static_cast<size_t>(bh) * R + r) * N + n;
        sBt[n * R + r] = to_f(Bt[o]);
        sCt[n * R + r] = to_f(Ct[o]);
      }
      if (i < R * P) sx[i] = to_f(xt[i]);
    }
    __syncthreads();
  }
  if constexpr (kNorm)
    row_inv_rms<Tin>(Bt + static_cast<size_t>(bh) * R * N, Ct + static_cast<size_t>(bh) * R * N,
                     prevB + static_cast<size_t>(bh) * R * N, R, N, q.neps, sinv);
  for (int i = threadIdx.x; kRot && (i < R * K || i < R * P); i += blockDim.x) {
    const bool rot = i < R * K, cpy = i < R * P;
    const int r = rot ? i / K : 0, k = rot ? i - r * K : 0;
    const size_t o = (static_cast<size_t>(bh) * R + r) * N + 2 * k;
    float ph0 = 0.f, thk = 0.f, pu = 0.f, pv = 0.f, cu = 0.f, cv = 0.f;
    Tin bu_raw{}, bv_raw{}, xv{};
    float xpv = 0.f;
    if (rot) {
      ph0 = p.phi[static_cast<size_t>(bh) * K + k];
      thk = to_f(th[k]);
      pu = to_f(prevB[o]);
      pv = to_f(prevB[o + 1]);
      bu_raw = Bt[o];
      bv_raw = Bt[o + 1];
      cu = to_f(Ct[o]);
      cv = to_f(Ct[o + 1]);
    }
    if (cpy) {
      xv = xt[i];
      xpv = to_f(prevx[i]);
    }
    if (rot) {
      const float ph1 = ph0 + dt * thk;
      float s0, c0, s1, c1;
      __sincosf(fmaf(-6.283185307179586f, rintf(ph0 * 0.15915494309189535f), ph0), &s0, &c0);
      __sincosf(fmaf(-6.283185307179586f, rintf(ph1 * 0.15915494309189535f), ph1), &s1, &c1);
      float bu = to_f(bu_raw), bv = to_f(bv_raw);
      if constexpr (kNorm) {  // BCNorm and bias before the rotation; prev_B is stored raw
        const Tin* nwB = static_cast<const Tin*>(q.nwB);
        const Tin* nwC = static_cast<const Tin*>(q.nwC);
        const Tin* nbB = q.nbB ? static_cast<const Tin*>(q.nbB) + static_cast<size_t>(head) * N : nullptr;
        const Tin* nbC = q.nbC ? static_cast<const Tin*>(q.nbC) + static_cast<size_t>(head) * N : nullptr;
        const int n0 = 2 * k, n1 = 2 * k + 1;
        const float wb0 = nwB ? to_f(nwB[n0]) : 1.f, wb1 = nwB ? to_f(nwB[n1]) : 1.f;
        const float bb0 = nbB ? to_f(nbB[n0]) : 0.f, bb1 = nbB ? to_f(nbB[n1]) : 0.f;
        const float wc0 = nwC ? to_f(nwC[n0]) : 1.f, wc1 = nwC ? to_f(nwC[n1]) : 1.f;
        const float bc0 = nbC ? to_f(nbC[n0]) : 0.f, bc1 = nbC ? to_f(nbC[n1]) : 0.f;
        const float ib = sinv[r], ic = sinv[R + r], ip = sinv[2 * R + r];
        bu = fmaf(bu * ib, wb0, bb0);
        bv = fmaf(bv * ib, wb1, bb1);
        cu = fmaf(cu * ic, wc0, bc0);
        cv = fmaf(cv * ic, wc1, bc1);
        pu = fmaf(pu * ip, wb0, bb0);
        pv = fmaf(pv * ip, wb1, bb1);
      }
      sBp[(2 * k) * R + r] = c0 * pu + s0 * pv;
      sBp[(2 * k + 1) * R + r] = -s0 * pu + c0 * pv;
      sBt[(2 * k) * R + r] = c1 * bu + s1 * bv;
      sBt[(2 * k + 1) * R + r] = -s1 * bu + c1 * bv;
      sCt[(2 * k) * R + r] = c1 * cu + s1 * cv;
      sCt[(2 * k + 1) * R + r] = -s1 * cu + c1 * cv;
      prevB[o] = bu_raw;
      prevB[o + 1] = bv_raw;
      if (r == 0) sphi[k] = ph1;  // written back after the barrier: other columns read phi
    }
    if (cpy) {
      sxp[i] = xpv;
      sx[i] = to_f(xv);
      prevx[i] = xv;
    }
  }
  if constexpr (kRot) __syncthreads();
  for (int k = threadIdx.x; kRot && k < K; k += blockDim.x)
    p.phi[static_cast<size_t>(bh) * K + k] =
        fmaf(-6.283185307179586f, rintf(sphi[k] * 0.15915494309189535f), sphi[k]);

  const float alpha = expf(dt * p.A[head]);
  const float beta = (1.f - lam) * dt * alpha;
  const float gamma = lam * dt;

  // The thread's column pair goes through packed f32x2 FMAs: per rank, one FMA each for
  // the previous-token and current-token products and one for the output.
  float2 xr[R], xpr[R], yp[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    xr[r] = *reinterpret_cast<const float2*>(&sx[r * P + 2 * cg]);
    xpr[r] = kRot ? *reinterpret_cast<const float2*>(&sxp[r * P + 2 * cg]) : make_float2(0.f, 0.f);
    yp[r] = make_float2(0.f, 0.f);
  }
  const float2 a2 = make_float2(alpha, alpha);

#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int n = rg + i * RG;
    float bp[R], bt[R], ct[R];
    if constexpr (kRot) load_r<R>(&sBp[n * R], bp);
    load_r<R>(&sBt[n * R], bt);
    load_r<R>(&sCt[n * R], ct);
    float2 prev = make_float2(0.f, 0.f), cur = make_float2(0.f, 0.f);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if constexpr (kRot) prev = __ffma2_rn(make_float2(beta * bp[r], beta * bp[r]), xpr[r], prev);
      cur = __ffma2_rn(make_float2(gamma * bt[r], gamma * bt[r]), xr[r], cur);
    }
    const float2 h = __ffma2_rn(a2, hv[i], __fadd2_rn(prev, cur));
#pragma unroll
    for (int r = 0; r < R; ++r) yp[r] = __ffma2_rn(h, make_float2(ct[r], ct[r]), yp[r]);
    __stcs(reinterpret_cast<float2*>(hs + static_cast<size_t>(n) * P) + cg, h);
  }

#pragma unroll
  for (int r = 0; r < R; ++r) *reinterpret_cast<float2*>(&red[(rg * R + r) * P + 2 * cg]) = yp[r];
  __syncthreads();

  Tout* y = static_cast<Tout*>(p.y) + static_cast<size_t>(bh) * R * P;
  for (int i = threadIdx.x; i < R * P; i += blockDim.x) {
    float acc = 0.f;
    for (int g = 0; g < RG; ++g) acc += red[g * R * P + i];
    from_f(y[i], acc);
  }
}

size_t smem_bytes(const m3_dims& d, int RG);

template <typename Tin, typename Tout, int R, bool kRot, bool kNorm>
cudaError_t launch_r(const DecodeArgs& a, cudaStream_t s, int threads, int vpt) {
  const m3_dims& d = a.d;
  DecodeParams p{a.s.h, a.s.phi, a.s.prev_B, a.s.prev_x, a.x, a.B, a.C, a.dt, a.A, a.lam, a.theta,
                 a.y, d.H, d.N, d.P};
  DecodeNorm q{a.norm ? a.norm->B_weight : nullptr, a.norm ? a.norm->B_bias : nullptr,
               a.norm ? a.norm->C_weight : nullptr, a.norm ? a.norm->C_bias : nullptr,
               a.norm ? a.norm->eps : 1.f};
  const int RG = threads / (d.P / 2);
  const size_t smem = smem_bytes(d, RG);
  const dim3 grid(static_cast<unsigned>(d.B) * static_cast<unsigned>(d.H));
  auto go = [&](auto k) -> cudaError_t {
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    k<<<grid, threads, smem, s>>>(p, q);
    return cudaGetLastError();
  };
  if (threads <= 256) {
    switch (vpt) {
      case 1: return go(decode_step_kernel<Tin, Tout, R, 1, 256, kRot, kNorm>);
      case 2: return go(decode_step_kernel<Tin, Tout, R, 2, 256, kRot, kNorm>);
      case 4: return go(decode_step_kernel<Tin, Tout, R, 4, 256, kRot, kNorm>);
      case 8: return go(decode_step_kernel<Tin, Tout, R, 8, 256, kRot, kNorm>);
      case 16: return go(decode_step_kernel<Tin, Tout, R, 16, 256, kRot, kNorm>);
      case 32: return go(decode_step_kernel<Tin, Tout, R, 32, 256, kRot, kNorm>);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (vpt) {
    case 8: return go(decode_step_kernel<Tin, Tout, R, 8, 1024, kRot, kNorm>);
    case 16: return go(decode_step_kernel<Tin, Tout, R, 16, 1024, kRot, kNorm>);
    case 32: return go(decode_step_kernel<Tin, Tout, R, 32, 1024, kRot, kNorm>);
    default: return cudaErrorInvalidValue;
  }
}

size_t smem_bytes(const m3_dims& d, int RG) {
  return sizeof(float) * (3 * d.R * d.N + 2 * d.R * d.P + RG * d.R * d.P + d.N / 2 + 3 * d.R);
}

// Each thread keeps VPT in {1,2,4,8,16,32} float2 of state (VPT divides N), so
// threads = (P/2) * (N / VPT).  Take the smallest VPT that gives at most 256
// threads; failing that, the smallest VPT >= 8 that fits 1024 threads.
bool plan(const m3_dims& d, int* threads, int* vpt) {
  if (d.P % 4 != 0 || d.P < 4 || d.N < 2) return false;
  const int P2 = d.P / 2;
  int fallback = 0;
  for (int v = 1; v <= 32; v *= 2) {
    if (d.N % v != 0) continue;
    const int t = P2 * (d.N / v);
    if (t > 1024 || smem_bytes(d, d.N / v) > 96 * 1024) continue;
    if (t <= 256) {
      *threads = t;
      *vpt = v;
      return true;
    }
    if (fallback == 0 && v >= 8) fallback = v;
  }
  if (fallback == 0) return false;
  *vpt = fallback;
  *threads = P2 * (d.N / fallback);
  return true;
}

}  // namespace

bool decode_supported(const m3_dims& d) {
  int t, v;
  return plan(d, &t, &v);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  int threads, vpt;
  if (!plan(a.d, &threads, &vpt)) return cudaErrorInvalidValue;
  const bool bf_in = a.d.in_dtype == M3_BF16, bf_out = a.d.out_dtype == M3_BF16;
  // No theta: the Mamba-2 special case, SISO only (state h alone).
  if (!a.theta) {
    if (a.d.R != 1 || a.lam || a.s.phi || a.s.prev_B || a.s.prev_x || a.norm)
      return cudaErrorInvalidValue;
    if (bf_in && bf_out) return launch_r<__nv_bfloat16, __nv_bfloat16, 1, false, false>(a, s, threads, vpt);
    if (bf_in) return launch_r<__nv_bfloat16, float, 1, false, false>(a, s, threads, vpt);
    if (bf_out) return launch_r<float, __nv_bfloat16, 1, false, false>(a, s, threads, vpt);
    return launch_r<float, float, 1, false, false>(a, s, threads, vpt);
  }
#define M3_RN(RR, NORM)                                                                                 \
  if (bf_in && bf_out) return launch_r<__nv_bfloat16, __nv_bfloat16, RR, true, NORM>(a, s, threads, vpt); \
  if (bf_in) return launch_r<__nv_bfloat16, float, RR, true, NORM>(a, s, threads, vpt);                   \
  if (bf_out) return launch_r<float, __nv_bfloat16, RR, true, NORM>(a, s, threads, vpt);                  \
  return launch_r<float, float, RR, true, NORM>(a, s, threads, vpt);
#define M3_R(RR)          \
  if (a.d.R == RR) {      \
    if (a.norm) {         \
      M3_RN(RR, true)     \
    } else {              \
      M3_RN(RR, false)    \
    }                     \
  }
  M3_R(1)
  M3_R(2)
  M3_R(4)
  M3_R(8)
#undef M3_R
#undef M3_RN
  return cudaErrorInvalidValue;
}

}  // namespace m3
