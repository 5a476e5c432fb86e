// Recurrent prefill on CUDA cores (fp32 arithmetic, any supported shape).
//
// Runs the exponential-trapezoidal recurrence of Proposition 1 token by token
// with the rotation of Proposition 3 and the MIMO rank-R products of section
// 3.3, one CTA per (batch row, head).  This is the path for fp32 inputs,
// whose tolerance (1e-4 of the output RMS) tensor-core tf32/bf16 operands
// cannot meet, and for shapes outside the tensor-core kernel's tiling.
//
// Thread (p, g) holds column p of rows g, g + G, ... of the N x P state in
// registers.  Per token: threads rotate B_t, C_t into shared memory (double
// buffered, so the previous token's rotated B stays available for the beta
// term), update their state entries, write partial outputs, and a fixed-order
// reduction over g produces y_t.  With no lambda and no theta (null pointers) the
// kernel runs the Mamba-2 special case, lambda = 1 and theta = 0.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "m3_internal.h"

namespace m3 {
namespace {

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ void from_f(float& d, float v) { d = v; }
__device__ __forceinline__ void from_f(__nv_bfloat16& d, float v) { d = __float2bfloat16_rn(v); }

constexpr int kMaxRows = 32;  // state rows per thread

struct RecParams {
  const void* x;
  const void* B;
  const void* C;
  const void* dt;
  const float* A;
  const void* lam;
  const void* theta;
  const float* h0;
  const float* phi0;
  const void* prevB0;
  const void* prevx0;
  void* y;
  float* hT;
  float* phiT;
  void* prevBT;
  void* prevxT;
  int T, H, N, P, R, G;
  // BCNorm + biases (section 3.4) of B, C and the stored raw previous B, when norm != 0:
  // weights [N] (null: ones), biases [H][N] (null: zeros), in the input dtype.
  int norm;
  const void* nwB;
  const void* nbB;
  const void* nwC;
  const void* nbC;
  float neps;
};

// 1 / RMS over the N entries of each of `rows` rows (row j starts at src(j)), into s_inv[j],
// in a fixed summation order.  Whole warps take one row each; a block that is not a whole
// number of warps uses one thread per row.  Ends with a barrier.
template <typename Tin, typename RowFn>
__device__ void rows_inv_rms(RowFn src, int rows, int N, float eps, float* s_inv) {
  if ((blockDim.x & 31) == 0) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    for (int j = warp; j < rows; j += nwarps) {
      const Tin* row = src(j);
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
    for (int j = threadIdx.x; j < rows; j += blockDim.x) {
      const Tin* row = src(j);
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

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(1024) prefill_recurrent_kernel(const RecParams p) {
  const int bh = blockIdx.x;
  const int b = bh / p.H, head = bh % p.H;
  const int T = p.T, H = p.H, N = p.N, P = p.P, R = p.R, G = p.G, K = N / 2;
  const int pcol = threadIdx.x % P;
  const int g = threadIdx.x / P;
  const int rows = N / G;

  extern __shared__ float sm[];
  float* sB = sm;                 // [2][R][N]  rotated B, by token parity
  float* sC = sB + 2 * R * N;     // [R][N]     rotated C of the current token
  float* sx = sC + R * N;         // [2][R][P]  x, by token parity
  float* red = sx + 2 * R * P;    // [G][R][P]
  float* sphi = red + G * R * P;  // [K]
  float* sinv = sphi + K;         // [2R] BCNorm 1/RMS of the token's B, C rows (or prev_B)

  const Tin* xg = static_cast<const Tin*>(p.x);
  const Tin* Bg = static_cast<const Tin*>(p.B);
  const Tin* Cg = static_cast<const Tin*>(p.C);
  const Tin* dtg = static_cast<const Tin*>(p.dt);
  const Tin* lamg = static_cast<const Tin*>(p.lam);
  const Tin* thg = static_cast<const Tin*>(p.theta);
  const float A = p.A[head];
  const Tin* nwB = static_cast<const Tin*>(p.nwB);
  const Tin* nbB = p.nbB ? static_cast<const Tin*>(p.nbB) + static_cast<size_t>(head) * N : nullptr;
  const Tin* nwC = static_cast<const Tin*>(p.nwC);
  const Tin* nbC = p.nbC ? static_cast<const Tin*>(p.nbC) + static_cast<size_t>(head) * N : nullptr;
  // BCNorm and the bias of element n of a row scaled by 1/RMS `inv` (weights w, biases c)
  auto nrm = [&](float v, float inv, const Tin* w, const Tin* c, int n) {
    return fmaf(v * inv, w ? to_f(w[n]) : 1.f, c ? to_f(c[n]) : 0.f);
  };
  if (p.norm && p.prevB0) {
    const Tin* pb0 = static_cast<const Tin*>(p.prevB0) + static_cast<size_t>(bh) * R * N;
    rows_inv_rms<Tin>([&](int j) { return pb0 + static_cast<size_t>(j) * N; }, R, N, p.neps, sinv);
  }

  // Entry state.  Slot 1 of the rotated-B / x buffers holds the previous token
  // (rotated by its own angle) because token 0 uses parity 0.
  float hreg[kMaxRows];
#pragma unroll
  for (int i = 0; i < kMaxRows; ++i) {
    const int n = g + i * G;
    hreg[i] = (i < rows && p.h0) ? p.h0[(static_cast<size_t>(bh) * N + n) * P + pcol] : 0.f;
  }
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    const float ph = p.phi0 ? p.phi0[static_cast<size_t>(bh) * K + k] : 0.f;
    sphi[k] = ph;
    float s, c;
    sincosf(ph, &s, &c);
    for (int r = 0; r < R; ++r) {
      float u = 0.f, v = 0.f;
      if (p.prevB0) {
        const Tin* pb = static_cast<const Tin*>(p.prevB0) + (static_cast<size_t>(bh) * R + r) * N;
        u = to_f(pb[2 * k]);
        v = to_f(pb[2 * k + 1]);
        if (p.norm) {  // the stored previous token is raw
          u = nrm(u, sinv[r], nwB, nbB, 2 * k);
          v = nrm(v, sinv[r], nwB, nbB, 2 * k + 1);
        }
      }
      sB[(R + r) * N + 2 * k] = c * u + s * v;
      sB[(R + r) * N + 2 * k + 1] = -s * u + c * v;
    }
  }
  for (int i = threadIdx.x; i < R * P; i += blockDim.x)
    sx[R * P + i] =
        p.prevx0 ? to_f(static_cast<const Tin*>(p.prevx0)[static_cast<size_t>(bh) * R * P + i])
                 : 0.f;
  __syncthreads();

  for (int t = 0; t < T; ++t) {
    const int cur = t & 1, prv = cur ^ 1;
    const size_t tok = (static_cast<size_t>(b) * T + t) * H + head;  // (b, t, head)
    const float dt = to_f(dtg[tok]);
    const float lam = lamg ? to_f(lamg[tok]) : 1.f;  // no lambda, no theta: the Mamba-2 case

    // 0. BCNorm: 1/RMS of the token's B and C rows (the barrier also ends the previous
    //    token's reads of sinv)
    if (p.norm)
      rows_inv_rms<Tin>([&](int j) { return (j < R ? Bg : Cg) + (tok * R + (j % R)) * N; }, 2 * R,
                        N, p.neps, sinv);
    // 1. advance the angle, rotate B_t and C_t; stage x_t.
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
      const float ph = thg ? sphi[k] + dt * to_f(thg[tok * K + k]) : sphi[k];
      sphi[k] = fmaf(-6.283185307179586f, rintf(ph * 0.15915494309189535f), ph);  // keep |phi| <= pi
      float s, c;
      sincosf(ph, &s, &c);
      for (int r = 0; r < R; ++r) {
        const size_t o = (tok * R + r) * N + 2 * k;
        float bu = to_f(Bg[o]), bv = to_f(Bg[o + 1]);
        float cu = to_f(Cg[o]), cv = to_f(Cg[o + 1]);
        if (p.norm) {
          bu = nrm(bu, sinv[r], nwB, nbB, 2 * k);
          bv = nrm(bv, sinv[r], nwB, nbB, 2 * k + 1);
          cu = nrm(cu, sinv[R + r], nwC, nbC, 2 * k);
          cv = nrm(cv, sinv[R + r], nwC, nbC, 2 * k + 1);
        }
        sB[(cur * R + r) * N + 2 * k] = c * bu + s * bv;
        sB[(cur * R + r) * N + 2 * k + 1] = -s * bu + c * bv;
        sC[r * N + 2 * k] = c * cu + s * cv;
        sC[r * N + 2 * k + 1] = -s * cu + c * cv;
      }
    }
    for (int i = threadIdx.x; i < R * P; i += blockDim.x) sx[cur * R * P + i] = to_f(xg[tok * R * P + i]);
    __syncthreads();

    // 2. state update and partial outputs.
    const float alpha = expf(dt * A);
    const float beta = (1.f - lam) * dt * alpha;
    const float gamma = lam * dt;
    float yp[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) yp[r] = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxRows; ++i) {
      if (i < rows) {
        const int n = g + i * G;
        float pterm = 0.f, cterm = 0.f;
        for (int r = 0; r < R; ++r) {
          pterm = fmaf(sB[(prv * R + r) * N + n], sx[(prv * R + r) * P + pcol], pterm);
          cterm = fmaf(sB[(cur * R + r) * N + n], sx[(cur * R + r) * P + pcol], cterm);
        }
        hreg[i] = fmaf(alpha, hreg[i], fmaf(beta, pterm, gamma * cterm));
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (r < R) yp[r] = fmaf(hreg[i], sC[r * N + n], yp[r]);
      }
    }
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (r < R) red[(g * R + r) * P + pcol] = yp[r];
    __syncthreads();

    // 3. y_t = sum over g, fixed order.
    Tout* yt = static_cast<Tout*>(p.y) + tok * R * P;
    for (int i = threadIdx.x; i < R * P; i += blockDim.x) {
      float acc = 0.f;
      for (int gg = 0; gg < G; ++gg) acc += red[gg * R * P + i];
      from_f(yt[i], acc);
    }
  }

  // Exit state (the entry state was read above, so hT may alias h0).
  if (p.hT) {
#pragma unroll
    for (int i = 0; i < kMaxRows; ++i)
      if (i < rows) p.hT[(static_cast<size_t>(bh) * N + g + i * G) * P + pcol] = hreg[i];
  }
  __syncthreads();
  if (p.phiT)
    for (int k = threadIdx.x; k < K; k += blockDim.x) p.phiT[static_cast<size_t>(bh) * K + k] = sphi[k];
  if (p.prevBT) {
    Tin* out = static_cast<Tin*>(p.prevBT) + static_cast<size_t>(bh) * R * N;
    for (int i = threadIdx.x; i < R * N; i += blockDim.x) {
      Tin v;
      if (T > 0)
        v = Bg[((static_cast<size_t>(b) * T + T - 1) * H + head) * R * N + i];
      else if (p.prevB0)
        v = static_cast<const Tin*>(p.prevB0)[static_cast<size_t>(bh) * R * N + i];
      else
        from_f(v, 0.f);
      out[i] = v;
    }
  }
  if (p.prevxT) {
    Tin* out = static_cast<Tin*>(p.prevxT) + static_cast<size_t>(bh) * R * P;
    for (int i = threadIdx.x; i < R * P; i += blockDim.x) {
      Tin v;
      if (T > 0)
        v = xg[((static_cast<size_t>(b) * T + T - 1) * H + head) * R * P + i];
      else if (p.prevx0)
        v = static_cast<const Tin*>(p.prevx0)[static_cast<size_t>(bh) * R * P + i];
      else
        from_f(v, 0.f);
      out[i] = v;
    }
  }
}

// G = number of row groups: the largest power of two that divides N with
// P * G <= 1024 threads, subject to N / G <= kMaxRows.
int plan_groups(const m3_dims& d) {
  int best = 0;
  for (int g = 1; g <= d.N && d.P * g <= 1024; g *= 2) {
    if (d.N % g != 0) break;
    if (d.N / g <= kMaxRows) best = g;
    if (best && d.P * g >= 256) break;
  }
  return best;
}

size_t rec_smem(const m3_dims& d, int G) {
  return sizeof(float) * (3 * d.R * d.N + 2 * d.R * d.P + G * d.R * d.P + d.N / 2 + 2 * d.R);
}

template <typename Tin, typename Tout>
cudaError_t launch_t(const PrefillArgs& a, cudaStream_t s) {
  const m3_dims& d = a.d;
  const int G = plan_groups(d);
  RecParams p{a.x,      a.B,         a.C,         a.dt,        a.A,         a.lam,
              a.theta,  a.h0.h,      a.h0.phi,    a.h0.prev_B, a.h0.prev_x, a.y,
              a.hT.h,   a.hT.phi,    a.hT.prev_B, a.hT.prev_x, d.T,         d.H,
              d.N,      d.P,         d.R,         G,
              a.norm ? 1 : 0,
              a.norm ? a.norm->B_weight : nullptr,
              a.norm ? a.norm->B_bias : nullptr,
              a.norm ? a.norm->C_weight : nullptr,
              a.norm ? a.norm->C_bias : nullptr,
              a.norm ? a.norm->eps : 1.f};
  const size_t smem = rec_smem(d, G);
  auto k = prefill_recurrent_kernel<Tin, Tout>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  k<<<static_cast<unsigned>(d.B) * static_cast<unsigned>(d.H), d.P * G, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool prefill_recurrent_supported(const m3_dims& d) {
  const int G = plan_groups(d);
  return G > 0 && rec_smem(d, G) <= 200 * 1024;
}

cudaError_t launch_prefill_recurrent(const PrefillArgs& a, cudaStream_t s) {
  const bool bi = a.d.in_dtype == M3_BF16, bo = a.d.out_dtype == M3_BF16;
  if (bi && bo) return launch_t<__nv_bfloat16, __nv_bfloat16>(a, s);
  if (bi) return launch_t<__nv_bfloat16, float>(a, s);
  if (bo) return launch_t<float, __nv_bfloat16>(a, s);
  return launch_t<float, float>(a, s);
}

}  // namespace m3
