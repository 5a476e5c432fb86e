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

// Threads: (P/4) column groups x RG row groups.  Thread (cg, rg) owns the
// float4 columns 4cg..4cg+3 of rows rg, rg + RG, ..., rg + (VPT-1) RG.
template <typename Tin, typename Tout, int R, int VPT>
__global__ void __launch_bounds__(1024) decode_step_kernel(const DecodeParams p) {
  const int bh = blockIdx.x;
  const int head = bh % p.H;
  const int N = p.N, P = p.P, K = N >> 1;
  const int P4 = P >> 2;
  const int cg = threadIdx.x % P4;
  const int rg = threadIdx.x / P4;
  const int RG = blockDim.x / P4;

  float* hs = p.h + static_cast<size_t>(bh) * N * P;
  float4 hv[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i)
    hv[i] = __ldcs(reinterpret_cast<const float4*>(hs + static_cast<size_t>(rg + i * RG) * P) + cg);

  extern __shared__ float sm[];
  float* sBt = sm;               // [R][N] B~_t
  float* sCt = sBt + R * N;      // [R][N] C~_t
  float* sBp = sCt + R * N;      // [R][N] B~_{t-1}
  float* sx = sBp + R * N;       // [R][P] X_t
  float* sxp = sx + R * P;       // [R][P] X_{t-1}
  float* red = sxp + R * P;      // [RG][R][P] partial outputs
  float* sphi = red + RG * R * P;  // [K] advanced angle

  const Tin* Bt = static_cast<const Tin*>(p.B);
  const Tin* Ct = static_cast<const Tin*>(p.C);
  Tin* prevB = static_cast<Tin*>(p.prevB);
  const float dt = to_f(static_cast<const Tin*>(p.dt)[bh]);
  const float lam = to_f(static_cast<const Tin*>(p.lam)[bh]);
  const Tin* th = static_cast<const Tin*>(p.theta) + static_cast<size_t>(bh) * K;

  // Rotations: previous token by its own angle phi, current token by phi + dt theta.
  // One thread per (rank column r, pair k), so the R columns rotate in parallel.
  for (int i = threadIdx.x; i < R * K; i += blockDim.x) {
    const int r = i / K, k = i - r * K;
    const float ph0 = p.phi[static_cast<size_t>(bh) * K + k];
    const float ph1 = ph0 + dt * to_f(th[k]);
    const size_t o = (static_cast<size_t>(bh) * R + r) * N + 2 * k;
    const float pu = to_f(prevB[o]), pv = to_f(prevB[o + 1]);
    const Tin bu_raw = Bt[o], bv_raw = Bt[o + 1];
    const float cu = to_f(Ct[o]), cv = to_f(Ct[o + 1]);
    const float bu = to_f(bu_raw), bv = to_f(bv_raw);
    float s0, c0, s1, c1;
    sincosf(ph0, &s0, &c0);
    sincosf(ph1, &s1, &c1);
    sBp[r * N + 2 * k] = c0 * pu + s0 * pv;
    sBp[r * N + 2 * k + 1] = -s0 * pu + c0 * pv;
    sBt[r * N + 2 * k] = c1 * bu + s1 * bv;
    sBt[r * N + 2 * k + 1] = -s1 * bu + c1 * bv;
    sCt[r * N + 2 * k] = c1 * cu + s1 * cv;
    sCt[r * N + 2 * k + 1] = -s1 * cu + c1 * cv;
    prevB[o] = bu_raw;
    prevB[o + 1] = bv_raw;
    if (r == 0) sphi[k] = ph1;  // written back after the barrier: other columns read phi
  }
  {
    const Tin* xt = static_cast<const Tin*>(p.x) + static_cast<size_t>(bh) * R * P;
    Tin* prevx = static_cast<Tin*>(p.prevx) + static_cast<size_t>(bh) * R * P;
    for (int i = threadIdx.x; i < R * P; i += blockDim.x) {
      sxp[i] = to_f(prevx[i]);
      const Tin v = xt[i];
      sx[i] = to_f(v);
      prevx[i] = v;
    }
  }
  __syncthreads();

  // stored reduced to [-pi, pi] so that long decode loops keep full precision
  for (int k = threadIdx.x; k < K; k += blockDim.x)
    p.phi[static_cast<size_t>(bh) * K + k] =
        fmaf(-6.283185307179586f, rintf(sphi[k] * 0.15915494309189535f), sphi[k]);

  const float alpha = expf(dt * p.A[head]);
  const float beta = (1.f - lam) * dt * alpha;
  const float gamma = lam * dt;

  float yp[R][4];
#pragma unroll
  for (int r = 0; r < R; ++r) yp[r][0] = yp[r][1] = yp[r][2] = yp[r][3] = 0.f;

#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int n = rg + i * RG;
    float hcur[4] = {hv[i].x, hv[i].y, hv[i].z, hv[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int pp = 4 * cg + j;
      float prev = 0.f, cur = 0.f;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        prev = fmaf(sBp[r * N + n], sxp[r * P + pp], prev);
        cur = fmaf(sBt[r * N + n], sx[r * P + pp], cur);
      }
      hcur[j] = fmaf(alpha, hcur[j], fmaf(beta, prev, gamma * cur));
#pragma unroll
      for (int r = 0; r < R; ++r) yp[r][j] = fmaf(hcur[j], sCt[r * N + n], yp[r][j]);
    }
    __stcs(reinterpret_cast<float4*>(hs + static_cast<size_t>(n) * P) + cg,
           make_float4(hcur[0], hcur[1], hcur[2], hcur[3]));
  }

#pragma unroll
  for (int r = 0; r < R; ++r)
    *reinterpret_cast<float4*>(&red[(rg * R + r) * P + 4 * cg]) =
        make_float4(yp[r][0], yp[r][1], yp[r][2], yp[r][3]);
  __syncthreads();

  Tout* y = static_cast<Tout*>(p.y) + static_cast<size_t>(bh) * R * P;
  for (int i = threadIdx.x; i < R * P; i += blockDim.x) {
    float acc = 0.f;
    for (int g = 0; g < RG; ++g) acc += red[g * R * P + i];
    from_f(y[i], acc);
  }
}

size_t smem_bytes(const m3_dims& d, int RG);

template <typename Tin, typename Tout, int R>
cudaError_t launch_r(const DecodeArgs& a, cudaStream_t s, int threads, int vpt) {
  const m3_dims& d = a.d;
  DecodeParams p{a.s.h, a.s.phi, a.s.prev_B, a.s.prev_x, a.x, a.B, a.C, a.dt, a.A, a.lam, a.theta,
                 a.y, d.H, d.N, d.P};
  const int RG = threads / (d.P / 4);
  const size_t smem = smem_bytes(d, RG);
  const dim3 grid(static_cast<unsigned>(d.B) * static_cast<unsigned>(d.H));
  switch (vpt) {
#define M3_CASE(V)                                                                             \
  case V: {                                                                                    \
    auto k = decode_step_kernel<Tin, Tout, R, V>;                                             \
    if (smem > 48 * 1024) {                                                                    \
      cudaError_t e =                                                                          \
          cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);    \
      if (e != cudaSuccess) return e;                                                          \
    }                                                                                          \
    k<<<grid, threads, smem, s>>>(p);                                                          \
    return cudaGetLastError();                                                                 \
  }
    M3_CASE(1)
    M3_CASE(2)
    M3_CASE(4)
    M3_CASE(8)
    M3_CASE(16)
#undef M3_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

size_t smem_bytes(const m3_dims& d, int RG) {
  return sizeof(float) * (3 * d.R * d.N + 2 * d.R * d.P + RG * d.R * d.P + d.N / 2);
}

// Each thread keeps VPT in {1,2,4,8,16} float4 of state (VPT divides N), so
// threads = (P/4) * (N / VPT).  Take the smallest VPT that gives at most 256
// threads; failing that, the smallest that fits 1024 threads.
bool plan(const m3_dims& d, int* threads, int* vpt) {
  if (d.P % 4 != 0 || d.P < 4 || d.N < 2) return false;
  const int P4 = d.P / 4;
  int fallback = 0;
  for (int v = 1; v <= 16; v *= 2) {
    if (d.N % v != 0) continue;
    const int t = P4 * (d.N / v);
    if (t > 1024 || smem_bytes(d, d.N / v) > 96 * 1024) continue;
    if (t <= 256) {
      *threads = t;
      *vpt = v;
      return true;
    }
    if (fallback == 0) fallback = v;
  }
  if (fallback == 0) return false;
  *vpt = fallback;
  *threads = P4 * (d.N / fallback);
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
#define M3_R(RR)                                                                                  \
  if (a.d.R == RR) {                                                                              \
    if (bf_in && bf_out) return launch_r<__nv_bfloat16, __nv_bfloat16, RR>(a, s, threads, vpt);  \
    if (bf_in) return launch_r<__nv_bfloat16, float, RR>(a, s, threads, vpt);                    \
    if (bf_out) return launch_r<float, __nv_bfloat16, RR>(a, s, threads, vpt);                   \
    return launch_r<float, float, RR>(a, s, threads, vpt);                                        \
  }
  M3_R(1)
  M3_R(2)
  M3_R(4)
  M3_R(8)
#undef M3_R
  return cudaErrorInvalidValue;
}

}  // namespace m3
