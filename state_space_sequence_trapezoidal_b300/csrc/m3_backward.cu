// Backward pass of the prefill: gradients of y (and of the exit state h_T) with respect to
// x, B, C, dt, A, lambda, theta and the entry state h, on CUDA cores in fp32.
//
// The forward map is the masked matrix form of Eq. (7) (section 2.3): within a chunk of c
// tokens, with chunk-local log-decay sums l_i = sum_{s<=i} dt_s A, trapezoid column weights
// w_s = gamma_s + q_{s+1} (q = (1 - lambda) dt, gamma = lambda dt) and the mask
//   Mh[i, s] = exp(l_i - l_s) w_s (s < i),  gamma_i (s = i),  0 (s > i),
// and the folded entry state Hp = H_in + q_0 B~_{-1}^T X_{-1} (the previous token's
// trapezoid term, B~ rotated by its own angle, Proposition 3), the states and outputs are
//   h_i = exp(l_i) Hp + sum_{s<=i} Mh[i, s] B~_s^T X_s,   Y_i = C~_i h_i.
// Its adjoint is the same masked form transposed.  With Gout the cotangent of the chunk's
// last state and Gh_i = C~_i^T dY_i (+ Gout at the last token):
//   dC~_i = exp(l_i) dY_i Hp^T + sum_s D[i, s] B~_s,          D[i, s] = Mh[i, s] dY_i X_s^T
//   dB~_s = sum_i D[i, s]^T C~_i + Mh[last, s] X_s Gout^T
//   dX_s  = sum_i Mh[i, s] (C~_i B~_s^T)^T dY_i + Mh[last, s] B~_s Gout
//   dHp   = sum_i exp(l_i) Gh_i   (= the cotangent of the previous chunk's last state)
//   dMh[i, s] = <C~_i B~_s^T, dY_i X_s^T> (+ <Gout, B~_s^T X_s> on the last row)
// then the chain rule through l, w, gamma, q, the fold and the rotation (dB = R(phi) dB~,
// d phi from the rotation's derivative, d theta_t = dt_t sum_{s>=t} d phi_s over the whole
// sequence).  MIMO rank R: rows are (token, rank) pairs and every rank pair of two tokens
// shares the tokens' mask entry.
//
// Three kernels:
//   bwd_scan_kernel      one CTA per (batch row, head): the chunk-level forward scan
//                        H_in(k+1) = exp(l_last) Hp(k) + sum_s Mh[last, s] B~_s^T X_s, storing
//                        every Hp(k) and the angle before every chunk, then the reverse scan
//                        G(k-1) = dHp(k) = exp(l_last) G(k) + sum_i exp(l_i) C~_i^T dY_i,
//                        storing every chunk's Gout.
//   bwd_chunk_kernel     one CTA per (batch row, head, chunk), all chunks in parallel: the
//                        adjoint above, the mask and fold parameters, the rotation adjoint and
//                        the chunk-local suffix sums of d phi.
//   bwd_finalize_kernel  one CTA per (batch row, head): adds the d phi of later chunks to
//                        d theta and d dt, and sums the per-(b, h) part of dA.
// A fourth kernel sums dA over batch rows.  Every reduction has a fixed order, so results are
// bit-identical from run to run.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "m3_internal.h"

namespace m3 {
namespace {

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

constexpr int kThreads = 256;
constexpr int kPad = 4;        // floats of padding at the end of each shared-memory row
constexpr int kMaxRows = 64;   // (token, rank) rows per chunk at most
constexpr int kMaxTok = 32;    // tokens per chunk at most (one warp lane each)

struct BwdParams {
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
  const void* dy;
  const float* dhT;
  float* dx;
  float* dB;
  float* dC;
  float* ddt;
  float* dlam;
  float* dtheta;
  float* dh0;
  float* wsPhi;   // [BH][nch][K]   angle of the token before chunk k, reduced to [-pi, pi]
  float* wsH;     // [BH][nch][N*P] folded entry state Hp(k)
  float* wsG;     // [BH][nch][N*P] cotangent of the state after the last token of chunk k
  float* wsDH0;   // [BH][N*P]      cotangent of Hp(0)
  float* wsSphi;  // [BH][nch][K]   sum of d phi over the chunk's tokens
  float* wsDa;    // [BH][nch]      sum over the chunk's tokens of d(dt A) * dt
  float* dApart;  // [BH]
  int T, H, N, P, R, c, M, nch, K;
};

__device__ __forceinline__ float wrap(float a) {
  return fmaf(-6.283185307179586f, rintf(a * 0.15915494309189535f), a);
}

// out(i, j, sum_k A(i, k) B(k, j)) for i < NI, j < NJ, with both operands in shared memory
// addressed by strides, A(i, k) = a[i * ai + k * ak] and B(k, j) = b[k * bk + j * bj]; TI x TJ
// outputs per thread, tiles dealt to the CTA's threads in order.  Reads past NI / NJ are
// clamped to the last row / column and their results dropped.
template <int TI, int TJ, typename FO>
__device__ __forceinline__ void sgemm(int NI, int NJ, int NK, const float* __restrict__ a, int ai,
                                      int ak, const float* __restrict__ b, int bk, int bj, FO out) {
  const int nti = (NI + TI - 1) / TI, ntj = (NJ + TJ - 1) / TJ;
  for (int tile = threadIdx.x; tile < nti * ntj; tile += blockDim.x) {
    const int i0 = (tile / ntj) * TI, j0 = (tile % ntj) * TJ;
    const float* ap[TI];
    const float* bp[TJ];
#pragma unroll
    for (int u = 0; u < TI; ++u) ap[u] = a + min(i0 + u, NI - 1) * ai;
#pragma unroll
    for (int v = 0; v < TJ; ++v) bp[v] = b + min(j0 + v, NJ - 1) * bj;
    float acc[TI][TJ];
#pragma unroll
    for (int u = 0; u < TI; ++u)
#pragma unroll
      for (int v = 0; v < TJ; ++v) acc[u][v] = 0.f;
#pragma unroll 4
    for (int k = 0; k < NK; ++k) {
      float av[TI], bv[TJ];
#pragma unroll
      for (int u = 0; u < TI; ++u) av[u] = ap[u][k * ak];
#pragma unroll
      for (int v = 0; v < TJ; ++v) bv[v] = bp[v][k * bk];
#pragma unroll
      for (int u = 0; u < TI; ++u)
#pragma unroll
        for (int v = 0; v < TJ; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
    }
#pragma unroll
    for (int u = 0; u < TI; ++u)
#pragma unroll
      for (int v = 0; v < TJ; ++v)
        if (i0 + u < NI && j0 + v < NJ) out(i0 + u, j0 + v, acc[u][v]);
  }
}

// dst(i) = src(i) for i < n, four loads in flight per thread before their stores.
template <typename FS, typename FD>
__device__ __forceinline__ void stage(int n, FS src, FD dst) {
  const int nt = blockDim.x;
  for (int base = threadIdx.x; base < n; base += 4 * nt) {
    float v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = base + u * nt < n ? src(base + u * nt) : 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (base + u * nt < n) dst(base + u * nt, v[u]);
  }
}

// Fixed-order sum over the CTA of one float per thread (scratch: blockDim.x floats).
__device__ float block_sum(float v, float* scratch) {
  __syncthreads();
  scratch[threadIdx.x] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float s = 0.f;
    for (int i = threadIdx.x; i < static_cast<int>(blockDim.x); i += 32) s += scratch[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (threadIdx.x == 0) scratch[0] = s;
  }
  __syncthreads();
  const float r = scratch[0];
  __syncthreads();
  return r;
}

// Per-token coefficients of one chunk (tokens t < nt; entries up to c zeroed): dt, lambda,
// the chunk-local log-decay sums l, exp(l), gamma and q.  Warp 0, one lane per token.
template <typename Tin>
__device__ void chunk_coefs(const BwdParams& p, const Tin* dtg, const Tin* lamg, size_t tok0,
                            size_t tok_stride, int nt, float A, float* s_dt, float* s_lam,
                            float* s_ell, float* s_el, float* s_gam, float* s_q) {
  if (threadIdx.x < 32) {
    const int t = threadIdx.x;
    const bool ok = t < nt;
    const float dt = ok ? to_f(dtg[tok0 + t * tok_stride]) : 0.f;
    const float lam = ok ? to_f(lamg[tok0 + t * tok_stride]) : 0.f;
    float ell = dt * A;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float v = __shfl_up_sync(0xffffffffu, ell, o);
      if (t >= o) ell += v;
    }
    if (t < p.c) {
      s_dt[t] = dt;
      s_lam[t] = lam;
      s_ell[t] = ell;
      s_el[t] = ok ? expf(ell) : 0.f;
      s_gam[t] = lam * dt;
      s_q[t] = (1.f - lam) * dt;
    }
  }
}

// theta of the chunk's tokens into s_th[c][K] (zero past nt).
template <typename Tin>
__device__ __forceinline__ void stage_theta(const Tin* thg, size_t tok0, size_t tok_stride, int nt,
                                            int c, int K, float* s_th) {
  stage(c * K, [&](int e) {
    const int t = e / K;
    return t < nt ? to_f(thg[(tok0 + static_cast<size_t>(t) * tok_stride) * K + (e - t * K)]) : 0.f;
  }, [&](int e, float v) { s_th[e] = v; });
}

// Angles of the chunk's tokens: phi_t = phi_before + sum_{u<=t} dt_u theta_u (theta staged in
// s_th), as cos / sin [c][K] of the angle reduced to [-pi, pi]; returns through s_phi the
// reduced angle of the chunk's last token.
__device__ void chunk_angles(int nt, int K, const float* s_dt, const float* s_th, float* s_phi,
                             float* s_cs, float* s_sn) {
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    float ph = s_phi[k];
    for (int t = 0; t < nt; ++t) {
      ph = wrap(fmaf(s_dt[t], s_th[t * K + k], ph));
      float sn, cs;
      __sincosf(ph, &sn, &cs);
      s_cs[t * K + k] = cs;
      s_sn[t * K + k] = sn;
    }
    s_phi[k] = ph;
  }
}

// Rows (token t < nt, rank r) of a [T][H][R][N] operand of this (b, h), rotated by the tokens'
// angles, into dst[M][ld]; rows of tokens >= nt are zero.
template <typename Tin>
__device__ void load_rotated(const Tin* src, size_t tok0, size_t tok_stride, int nt, int R,
                             int N, int K, int M, const float* s_cs, const float* s_sn,
                             float* dst, int ld) {
  // raw rows first (several loads in flight per thread), then the rotation in place
  stage(M * N, [&](int e) {
    const int row = e / N, t = row / R;
    return t < nt ? to_f(src[((tok0 + static_cast<size_t>(t) * tok_stride) * R + (row - t * R)) * N + (e - row * N)])
                  : 0.f;
  }, [&](int e, float v) { dst[(e / N) * ld + e % N] = v; });
  __syncthreads();
  for (int e = threadIdx.x; e < M * K; e += blockDim.x) {
    const int row = e / K, k = e - row * K, t = row / R;
    const float u = dst[row * ld + 2 * k], v = dst[row * ld + 2 * k + 1];
    const float cs = t < nt ? s_cs[t * K + k] : 1.f, sn = t < nt ? s_sn[t * K + k] : 0.f;
    dst[row * ld + 2 * k] = cs * u + sn * v;
    dst[row * ld + 2 * k + 1] = -sn * u + cs * v;
  }
}

// Rows of a [T][H][R][P] operand into dst[M][ld] (zero past nt tokens).
template <typename T>
__device__ void load_rows(const T* src, size_t tok0, size_t tok_stride, int nt, int R, int P, int M,
                          float* dst, int ld) {
  stage(M * P, [&](int e) {
    const int row = e / P, t = row / R;
    return t < nt ? to_f(src[((tok0 + static_cast<size_t>(t) * tok_stride) * R + (row - t * R)) * P + (e - row * P)])
                  : 0.f;
  }, [&](int e, float v) { dst[(e / P) * ld + e % P] = v; });
}

// ------------------------------------------------------------------ shared-memory plans
struct ScanSmem {
  int H, BC, XY, th, cs, sn, prevB, prevX, phi, dt, lam, ell, el, gam, q, rs, red, total;
};
__host__ __device__ inline ScanSmem scan_smem(int N, int P, int R, int c) {
  const int K = N / 2, M = c * R;
  ScanSmem s{};
  int o = 0;
  auto take = [&](int n) {
    const int at = o;
    o += (n + 3) & ~3;
    return at;
  };
  s.H = take(N * (P + kPad));
  s.BC = take(M * (N + kPad));
  s.XY = take(M * (P + kPad));
  s.th = take(c * K);
  s.cs = take(c * K);
  s.sn = take(c * K);
  s.prevB = take(R * N);
  s.prevX = take(R * P);
  s.phi = take(K);
  s.dt = take(kMaxTok);
  s.lam = take(kMaxTok);
  s.ell = take(kMaxTok);
  s.el = take(kMaxTok);
  s.gam = take(kMaxTok);
  s.q = take(kMaxTok);
  s.rs = take(kMaxTok);
  s.red = take(kThreads);
  s.total = o;
  return s;
}

struct ChunkSmem {
  int Bt, Ct, X, dY, Hp, Go, S, E, W, dCt, dBt, dphi, dM, Mh, ex, rowel, wx, th, cs, sn, prevB,
      prevX, phi, dt, lam, ell, el, gam, q, dexp, dgam, dq, dell, red, total;
};
__host__ __device__ inline ChunkSmem chunk_smem(int N, int P, int R, int c) {
  const int K = N / 2, M = c * R;
  ChunkSmem s{};
  int o = 0;
  auto take = [&](int n) {
    const int at = o;
    o += (n + 3) & ~3;
    return at;
  };
  s.Bt = take(M * (N + kPad));   // B~
  s.Ct = take(M * (N + kPad));   // C~
  s.X = take(M * (P + kPad));
  s.dY = take(M * (P + kPad));
  s.Hp = take(N * (P + kPad));   // Hp
  s.Go = take(N * (P + kPad));   // Gout
  s.S = take(M * (M + kPad));    // C~ B~^T, then Mh o S
  s.E = take(M * (M + kPad));    // dY X^T, then Mh o E
  s.W = take(M * (P + kPad));    // B~ Gout
  s.dCt = take(M * (N + kPad));  // dY Hp^T, then dC~
  // dB~ [M][N + kPad] takes Hp's place once Hp is no longer read, where it fits
  s.dBt = N * (P + kPad) >= M * (N + kPad) ? s.Hp : take(M * (N + kPad));
  s.dphi = take(c * K);          // d phi per (token, pair), then its chunk-local suffix sums
  s.dM = take(kMaxTok * (kMaxTok + 1));
  s.Mh = take(kMaxTok * (kMaxTok + 1));   // Mh per token pair
  s.ex = take(kMaxTok * (kMaxTok + 1));   // exp(l_i - l_s) per token pair
  s.rowel = take(kMaxRows);               // exp(l) of each row's token
  s.wx = take(kMaxRows);                  // each row's weight on the exit-state terms
  s.th = take(c * K);
  s.cs = take(c * K);
  s.sn = take(c * K);
  s.prevB = take(R * N);
  s.prevX = take(R * P);
  s.phi = take(K);
  s.dt = take(kMaxTok);
  s.lam = take(kMaxTok);
  s.ell = take(kMaxTok);
  s.el = take(kMaxTok);
  s.gam = take(kMaxTok);
  s.q = take(kMaxTok + 1);
  s.dexp = take(kMaxTok);
  s.dgam = take(kMaxTok);
  s.dq = take(kMaxTok);
  s.dell = take(kMaxTok);
  s.red = take(kThreads);
  s.total = o;
  return s;
}

// ------------------------------------------------------------------ chunk-level scans
template <typename Tin, typename Tdy>
__global__ void __launch_bounds__(kThreads) bwd_scan_kernel(const BwdParams p) {
  extern __shared__ float sm[];
  const int bh = blockIdx.x, b = bh / p.H, head = bh % p.H;
  const int N = p.N, P = p.P, R = p.R, c = p.c, M = p.M, K = p.K, NP = N * P;
  const ScanSmem L = scan_smem(N, P, R, c);
  float* sH = sm + L.H;
  float* sBC = sm + L.BC;
  float* sXY = sm + L.XY;
  float* s_th = sm + L.th;
  float* s_cs = sm + L.cs;
  float* s_sn = sm + L.sn;
  float* s_pB = sm + L.prevB;
  float* s_pX = sm + L.prevX;
  float* s_phi = sm + L.phi;
  float* s_dt = sm + L.dt;
  float* s_lam = sm + L.lam;
  float* s_ell = sm + L.ell;
  float* s_el = sm + L.el;
  float* s_gam = sm + L.gam;
  float* s_q = sm + L.q;
  float* s_rs = sm + L.rs;
  const int ldN = N + kPad, ldP = P + kPad;
  const size_t tok_stride = p.H;
  const size_t seq0 = static_cast<size_t>(b) * p.T * p.H + head;
  const Tin* Bg = static_cast<const Tin*>(p.B);
  const Tin* Cg = static_cast<const Tin*>(p.C);
  const Tin* xg = static_cast<const Tin*>(p.x);
  const Tin* dtg = static_cast<const Tin*>(p.dt);
  const Tin* lamg = static_cast<const Tin*>(p.lam);
  const Tin* thg = static_cast<const Tin*>(p.theta);
  const Tdy* dyg = static_cast<const Tdy*>(p.dy);
  const float A = p.A[head];

  // entry state, angle and previous token (rotated by its own angle)
  for (int e = threadIdx.x; e < NP; e += blockDim.x)
    sH[(e / P) * ldP + e % P] = p.h0 ? p.h0[static_cast<size_t>(bh) * NP + e] : 0.f;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    const float ph = p.phi0 ? wrap(p.phi0[static_cast<size_t>(bh) * K + k]) : 0.f;
    s_phi[k] = ph;
    float sn, cs;
    sincosf(ph, &sn, &cs);
    for (int r = 0; r < R; ++r) {
      float u = 0.f, v = 0.f;
      if (p.prevB0) {
        const Tin* q = static_cast<const Tin*>(p.prevB0) + (static_cast<size_t>(bh) * R + r) * N + 2 * k;
        u = to_f(q[0]);
        v = to_f(q[1]);
      }
      s_pB[r * N + 2 * k] = cs * u + sn * v;
      s_pB[r * N + 2 * k + 1] = -sn * u + cs * v;
    }
  }
  for (int e = threadIdx.x; e < R * P; e += blockDim.x)
    s_pX[e] = p.prevx0 ? to_f(static_cast<const Tin*>(p.prevx0)[static_cast<size_t>(bh) * R * P + e]) : 0.f;
  __syncthreads();

  // ---------------------------------------------------------------- forward over chunks
  for (int k = 0; k < p.nch; ++k) {
    const int t0 = k * c, nt = min(c, p.T - t0);
    const size_t tok0 = seq0 + static_cast<size_t>(t0) * tok_stride;
    for (int kk = threadIdx.x; kk < K; kk += blockDim.x)
      p.wsPhi[(static_cast<size_t>(bh) * p.nch + k) * K + kk] = s_phi[kk];
    chunk_coefs<Tin>(p, dtg, lamg, tok0, tok_stride, nt, A, s_dt, s_lam, s_ell, s_el, s_gam, s_q);
    stage_theta<Tin>(thg, tok0, tok_stride, nt, c, K, s_th);
    __syncthreads();
    chunk_angles(nt, K, s_dt, s_th, s_phi, s_cs, s_sn);
    __syncthreads();
    load_rotated<Tin>(Bg, tok0, tok_stride, nt, R, N, K, M, s_cs, s_sn, sBC, ldN);
    load_rows<Tin>(xg, tok0, tok_stride, nt, R, P, M, sXY, ldP);
    // Hp = H + q_0 B~_prev^T X_prev, stored
    const float q0 = s_q[0];
    float* hp = p.wsH + (static_cast<size_t>(bh) * p.nch + k) * NP;
    for (int e = threadIdx.x; e < NP; e += blockDim.x) {
      const int n = e / P, pc = e - n * P;
      float f = 0.f;
      for (int r = 0; r < R; ++r) f = fmaf(s_pB[r * N + n], s_pX[r * P + pc], f);
      const float v = fmaf(q0, f, sH[n * ldP + pc]);
      sH[n * ldP + pc] = v;
      hp[e] = v;
    }
    __syncthreads();
    // the chunk's last token becomes the previous token of the next chunk (unscaled copy)
    const int last = nt - 1;
    for (int e = threadIdx.x; e < R * N; e += blockDim.x) s_pB[e] = sBC[(last * R + e / N) * ldN + e % N];
    for (int e = threadIdx.x; e < R * P; e += blockDim.x) s_pX[e] = sXY[(last * R + e / P) * ldP + e % P];
    // rows of B~ scaled by their token's Mh[last, token]
    if (threadIdx.x < c) {
      const int t = threadIdx.x;
      s_rs[t] = t > last ? 0.f
              : t == last ? s_gam[t]
                          : expf(s_ell[last] - s_ell[t]) * (s_gam[t] + s_q[t + 1]);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < M * N; e += blockDim.x) sBC[(e / N) * ldN + e % N] *= s_rs[(e / N) / R];
    __syncthreads();
    // H <- exp(l_last) Hp + sum_s Mh[last, s] B~_s^T X_s
    const float e_last = s_el[last];
    sgemm<4, 4>(N, P, M, sBC, 1, ldN, sXY, ldP, 1,
                [&](int n, int pc, float v) { sH[n * ldP + pc] = fmaf(e_last, sH[n * ldP + pc], v); });
    __syncthreads();
  }

  // ---------------------------------------------------------------- reverse over chunks
  for (int e = threadIdx.x; e < NP; e += blockDim.x)
    sH[(e / P) * ldP + e % P] = p.dhT ? p.dhT[static_cast<size_t>(bh) * NP + e] : 0.f;
  __syncthreads();
  for (int k = p.nch - 1; k >= 0; --k) {
    const int t0 = k * c, nt = min(c, p.T - t0);
    const size_t tok0 = seq0 + static_cast<size_t>(t0) * tok_stride;
    for (int kk = threadIdx.x; kk < K; kk += blockDim.x)
      s_phi[kk] = p.wsPhi[(static_cast<size_t>(bh) * p.nch + k) * K + kk];
    chunk_coefs<Tin>(p, dtg, lamg, tok0, tok_stride, nt, A, s_dt, s_lam, s_ell, s_el, s_gam, s_q);
    stage_theta<Tin>(thg, tok0, tok_stride, nt, c, K, s_th);
    __syncthreads();
    chunk_angles(nt, K, s_dt, s_th, s_phi, s_cs, s_sn);
    __syncthreads();
    load_rotated<Tin>(Cg, tok0, tok_stride, nt, R, N, K, M, s_cs, s_sn, sBC, ldN);
    load_rows<Tdy>(dyg, tok0, tok_stride, nt, R, P, M, sXY, ldP);
    float* go = p.wsG + (static_cast<size_t>(bh) * p.nch + k) * NP;
    for (int e = threadIdx.x; e < NP; e += blockDim.x) go[e] = sH[(e / P) * ldP + e % P];
    __syncthreads();
    // rows of C~ scaled by exp(l) of their token
    for (int e = threadIdx.x; e < M * N; e += blockDim.x) sBC[(e / N) * ldN + e % N] *= s_el[(e / N) / R];
    __syncthreads();
    // G <- exp(l_last) G + sum_i exp(l_i) C~_i^T dY_i
    const float e_last = s_el[nt - 1];
    sgemm<4, 4>(N, P, M, sBC, 1, ldN, sXY, ldP, 1,
                [&](int n, int pc, float v) { sH[n * ldP + pc] = fmaf(e_last, sH[n * ldP + pc], v); });
    __syncthreads();
  }
  for (int e = threadIdx.x; e < NP; e += blockDim.x) {
    const float v = sH[(e / P) * ldP + e % P];
    p.wsDH0[static_cast<size_t>(bh) * NP + e] = v;
    if (p.dh0) p.dh0[static_cast<size_t>(bh) * NP + e] = v;
  }
}

// ------------------------------------------------------------------ per-chunk adjoint
template <typename Tin, typename Tdy>
__global__ void __launch_bounds__(kThreads) bwd_chunk_kernel(const BwdParams p) {
  extern __shared__ float sm[];
  const int bh = blockIdx.x / p.nch, k = blockIdx.x % p.nch;
  const int b = bh / p.H, head = bh % p.H;
  const int N = p.N, P = p.P, R = p.R, c = p.c, M = p.M, K = p.K, NP = N * P;
  const ChunkSmem L = chunk_smem(N, P, R, c);
  float* sBt = sm + L.Bt;
  float* sCt = sm + L.Ct;
  float* sX = sm + L.X;
  float* sdY = sm + L.dY;
  float* sHp = sm + L.Hp;
  float* sdBt = sm + L.dBt;  // may share Hp's buffer: written only after Hp's last read
  float* sGo = sm + L.Go;
  float* sS = sm + L.S;
  float* sdphi = sm + L.dphi;
  float* sE = sm + L.E;
  float* sW = sm + L.W;
  float* sdCt = sm + L.dCt;
  float* s_dM = sm + L.dM;
  float* s_Mh = sm + L.Mh;
  float* s_ex = sm + L.ex;
  float* s_rowel = sm + L.rowel;
  float* s_wx = sm + L.wx;
  float* s_th = sm + L.th;
  float* s_cs = sm + L.cs;
  float* s_sn = sm + L.sn;
  float* s_pB = sm + L.prevB;
  float* s_pX = sm + L.prevX;
  float* s_phi = sm + L.phi;
  float* s_dt = sm + L.dt;
  float* s_lam = sm + L.lam;
  float* s_ell = sm + L.ell;
  float* s_el = sm + L.el;
  float* s_gam = sm + L.gam;
  float* s_q = sm + L.q;
  float* s_dexp = sm + L.dexp;
  float* s_dgam = sm + L.dgam;
  float* s_dq = sm + L.dq;
  float* s_dell = sm + L.dell;
  float* s_red = sm + L.red;
  const int ldN = N + kPad, ldP = P + kPad, ldM = M + kPad, ldT = kMaxTok + 1;
  const size_t tok_stride = p.H;
  const int t0 = k * c, nt = min(c, p.T - t0), last = nt - 1;
  const size_t seq0 = static_cast<size_t>(b) * p.T * p.H + head;
  const size_t tok0 = seq0 + static_cast<size_t>(t0) * tok_stride;
  const Tin* Bg = static_cast<const Tin*>(p.B);
  const Tin* Cg = static_cast<const Tin*>(p.C);
  const Tin* xg = static_cast<const Tin*>(p.x);
  const Tin* dtg = static_cast<const Tin*>(p.dt);
  const Tin* lamg = static_cast<const Tin*>(p.lam);
  const Tin* thg = static_cast<const Tin*>(p.theta);
  const Tdy* dyg = static_cast<const Tdy*>(p.dy);
  const float A = p.A[head];
  const bool has_next = k + 1 < p.nch;

  // ---------------------------------------------------------------- inputs of the chunk
  const float* phib = p.wsPhi + (static_cast<size_t>(bh) * p.nch + k) * K;
  for (int kk = threadIdx.x; kk < K; kk += blockDim.x) s_phi[kk] = phib[kk];
  chunk_coefs<Tin>(p, dtg, lamg, tok0, tok_stride, nt, A, s_dt, s_lam, s_ell, s_el, s_gam, s_q);
  if (threadIdx.x == 0) {  // q of the next chunk's first token (its fold weighs our last token)
    const size_t tn = tok0 + static_cast<size_t>(nt) * tok_stride;
    s_q[kMaxTok] = has_next ? (1.f - to_f(lamg[tn])) * to_f(dtg[tn]) : 0.f;
  }
  // the previous token (the previous chunk's last, or the entry state's), rotated by its angle
  for (int kk = threadIdx.x; kk < K; kk += blockDim.x) {
    float sn, cs;
    sincosf(phib[kk], &sn, &cs);
    for (int r = 0; r < R; ++r) {
      float u = 0.f, v = 0.f;
      if (k > 0) {
        const Tin* q = Bg + ((tok0 - tok_stride) * R + r) * N + 2 * kk;
        u = to_f(q[0]);
        v = to_f(q[1]);
      } else if (p.prevB0) {
        const Tin* q = static_cast<const Tin*>(p.prevB0) + (static_cast<size_t>(bh) * R + r) * N + 2 * kk;
        u = to_f(q[0]);
        v = to_f(q[1]);
      }
      s_pB[r * N + 2 * kk] = cs * u + sn * v;
      s_pB[r * N + 2 * kk + 1] = -sn * u + cs * v;
    }
  }
  for (int e = threadIdx.x; e < R * P; e += blockDim.x) {
    float v = 0.f;
    if (k > 0) v = to_f(xg[(tok0 - tok_stride) * R * P + e]);
    else if (p.prevx0) v = to_f(static_cast<const Tin*>(p.prevx0)[static_cast<size_t>(bh) * R * P + e]);
    s_pX[e] = v;
  }
  stage_theta<Tin>(thg, tok0, tok_stride, nt, c, K, s_th);
  __syncthreads();
  chunk_angles(nt, K, s_dt, s_th, s_phi, s_cs, s_sn);
  __syncthreads();
  load_rotated<Tin>(Bg, tok0, tok_stride, nt, R, N, K, M, s_cs, s_sn, sBt, ldN);
  load_rotated<Tin>(Cg, tok0, tok_stride, nt, R, N, K, M, s_cs, s_sn, sCt, ldN);
  load_rows<Tin>(xg, tok0, tok_stride, nt, R, P, M, sX, ldP);
  load_rows<Tdy>(dyg, tok0, tok_stride, nt, R, P, M, sdY, ldP);
  const float* hp = p.wsH + (static_cast<size_t>(bh) * p.nch + k) * NP;
  const float* go = p.wsG + (static_cast<size_t>(bh) * p.nch + k) * NP;
  stage(NP, [&](int e) { return hp[e]; }, [&](int e, float v) { sHp[(e / P) * ldP + e % P] = v; });
  stage(NP, [&](int e) { return go[e]; }, [&](int e, float v) { sGo[(e / P) * ldP + e % P] = v; });
  __syncthreads();

  // tables of the chunk: exp(l_i - l_s) and the mask Mh[i, s] per token pair; per row, exp(l)
  // of its token and its weight on the exit-state terms, Mh[last, s] plus q of the next
  // chunk's first token for the rows of the last token (their trapezoid term is folded into
  // the next chunk)
  const float q_next = s_q[kMaxTok];
  for (int e = threadIdx.x; e < c * c; e += blockDim.x) {
    const int ti = e / c, ts = e - ti * c;
    float ex = 0.f, m = 0.f;
    if (ts <= ti && ti < nt) {
      ex = expf(s_ell[ti] - s_ell[ts]);
      m = ts == ti ? s_gam[ti] : ex * (s_gam[ts] + s_q[ts + 1]);
    }
    s_ex[ti * ldT + ts] = ex;
    s_Mh[ti * ldT + ts] = m;
  }
  __syncthreads();
  for (int row = threadIdx.x; row < M; row += blockDim.x) {
    const int t = row / R;
    s_rowel[row] = s_el[t];
    s_wx[row] = t < nt ? s_Mh[last * ldT + t] + (t == last && has_next ? q_next : 0.f) : 0.f;
  }

  // ---------------------------------------------------------------- S, E, W = B~ Gout
  sgemm<2, 4>(M, M, N, sCt, ldN, 1, sBt, 1, ldN, [&](int i, int s_, float v) { sS[i * ldM + s_] = v; });
  sgemm<2, 4>(M, M, P, sdY, ldP, 1, sX, 1, ldP, [&](int i, int s_, float v) { sE[i * ldM + s_] = v; });
  sgemm<2, 4>(M, P, N, sBt, ldN, 1, sGo, ldP, 1, [&](int s_, int pc, float v) { sW[s_ * ldP + pc] = v; });
  // <Gout, Hp>
  float gh = 0.f;
  for (int e = threadIdx.x; e < NP; e += blockDim.x) gh = fmaf(sGo[(e / P) * ldP + e % P], sHp[(e / P) * ldP + e % P], gh);
  const float go_hp = block_sum(gh, s_red);  // (includes a barrier)

  // ---------------------------------------------------------------- dMh per token pair
  for (int e = threadIdx.x; e < c * c; e += blockDim.x) {
    const int ti = e / c, ts = e - ti * c;
    float v = 0.f;
    if (ts <= ti && ti < nt) {
      for (int r = 0; r < R; ++r)
        for (int r2 = 0; r2 < R; ++r2) v = fmaf(sS[(ti * R + r) * ldM + ts * R + r2], sE[(ti * R + r) * ldM + ts * R + r2], v);
      if (ti == last)  // the exit cotangent: <Gout, B~_s^T X_s>
        for (int r2 = 0; r2 < R; ++r2)
          for (int pc = 0; pc < P; ++pc) v = fmaf(sW[(ts * R + r2) * ldP + pc], sX[(ts * R + r2) * ldP + pc], v);
    }
    s_dM[ti * ldT + ts] = v;
  }
  __syncthreads();
  // Mh o S and Mh o E in place
  for (int e = threadIdx.x; e < M * M; e += blockDim.x) {
    const int i = e / M, s_ = e - i * M;
    const float m = s_Mh[(i / R) * ldT + s_ / R];
    sS[i * ldM + s_] *= m;
    sE[i * ldM + s_] *= m;
  }
  // Q = dY Hp^T into dC~
  sgemm<2, 4>(M, N, P, sdY, ldP, 1, sHp, 1, ldP, [&](int i, int n, float v) { sdCt[i * ldN + n] = v; });
  __syncthreads();
  // d exp(l_t) = sum over the token's rows of <C~_i, Q_i> (+ <Gout, Hp> at the last token)
  for (int t = threadIdx.x; t < c; t += blockDim.x) {
    float v = 0.f;
    if (t < nt)
      for (int r = 0; r < R; ++r)
        for (int n = 0; n < N; ++n) v = fmaf(sCt[(t * R + r) * ldN + n], sdCt[(t * R + r) * ldN + n], v);
    if (t == last) v += go_hp;
    s_dexp[t] = v;
  }
  __syncthreads();  // Q read; Hp no longer read (dB~ may take its buffer)
  // dC~ = D B~ + exp(l) Q
  sgemm<2, 4>(M, N, M, sE, ldM, 1, sBt, ldN, 1,
              [&](int i, int n, float v) { sdCt[i * ldN + n] = fmaf(s_rowel[i], sdCt[i * ldN + n], v); });
  // dB~ = D^T C~ + wexit(s) X_s Gout^T  (the same thread owns an output in both products)
  sgemm<2, 4>(M, N, M, sE, 1, ldM, sCt, ldN, 1, [&](int s_, int n, float v) { sdBt[s_ * ldN + n] = v; });
  sgemm<2, 4>(M, N, P, sX, ldP, 1, sGo, 1, ldP,
              [&](int s_, int n, float v) { sdBt[s_ * ldN + n] = fmaf(s_wx[s_], v, sdBt[s_ * ldN + n]); });
  // dX = (Mh o S)^T dY + wexit(s) W_s  -> global
  float* dxg = p.dx;
  sgemm<2, 4>(M, P, M, sS, 1, ldM, sdY, ldP, 1, [&](int s_, int pc, float v) {
    const int ts = s_ / R;
    if (ts < nt)
      dxg[(tok0 + static_cast<size_t>(ts) * tok_stride) * R * P + (s_ - ts * R) * P + pc] =
          fmaf(s_wx[s_], sW[s_ * ldP + pc], v);
  });
  // the fold of this chunk's entry: dq_0 += <dHp(k), B~_prev^T X_prev>, dHp(k) = Gout(k - 1)
  const float* dhp = k > 0 ? p.wsG + (static_cast<size_t>(bh) * p.nch + k - 1) * NP
                           : p.wsDH0 + static_cast<size_t>(bh) * NP;
  float fq = 0.f;
  stage(NP, [&](int e) { return dhp[e]; }, [&](int e, float v) {
    const int n = e / P, pc = e - n * P;
    float f = 0.f;
    for (int r = 0; r < R; ++r) f = fmaf(s_pB[r * N + n], s_pX[r * P + pc], f);
    fq = fmaf(v, f, fq);
  });
  const float dq_fold = block_sum(fq, s_red);  // (includes a barrier)

  // ---------------------------------------------------------------- mask and fold parameters
  if (threadIdx.x < c) {
    const int t = threadIdx.x;
    float dell = 0.f, dgam = 0.f, dq = 0.f;
    if (t < nt) {
      dell = s_dexp[t] * s_el[t];
      for (int ts = 0; ts < t; ++ts) dell = fmaf(s_dM[t * ldT + ts], s_Mh[t * ldT + ts], dell);  // row t
      for (int ti = t + 1; ti < nt; ++ti) {  // column t: l_t, gamma_t, q_{t+1}
        dell = fmaf(-s_dM[ti * ldT + t], s_Mh[ti * ldT + t], dell);
        dgam = fmaf(s_dM[ti * ldT + t], s_ex[ti * ldT + t], dgam);
      }
      dgam += s_dM[t * ldT + t];
      if (t == 0) {
        dq = dq_fold;
      } else {  // q_t weighs column t - 1
        for (int ti = t; ti < nt; ++ti) dq = fmaf(s_dM[ti * ldT + t - 1], s_ex[ti * ldT + t - 1], dq);
      }
    }
    s_dell[t] = dell;
    s_dgam[t] = dgam;
    s_dq[t] = dq;
  }
  __syncthreads();

  // ---------------------------------------------------------------- rotation adjoint, d phi
  for (int e = threadIdx.x; e < c * K; e += blockDim.x) sdphi[e] = 0.f;
  __syncthreads();
  float* dBg = p.dB;
  float* dCg = p.dC;
  // one thread per (token, pair): its R rows in a fixed order
  for (int e = threadIdx.x; e < nt * K; e += blockDim.x) {
    const int t = e / K, kk = e - t * K;
    const float cs = s_cs[t * K + kk], sn = s_sn[t * K + kk];
    float dph = 0.f;
    for (int r = 0; r < R; ++r) {
      const int row = t * R + r;
      const float db0 = sdBt[row * ldN + 2 * kk], db1 = sdBt[row * ldN + 2 * kk + 1];
      const float dc0 = sdCt[row * ldN + 2 * kk], dc1 = sdCt[row * ldN + 2 * kk + 1];
      const float b0 = sBt[row * ldN + 2 * kk], b1 = sBt[row * ldN + 2 * kk + 1];
      const float c0 = sCt[row * ldN + 2 * kk], c1 = sCt[row * ldN + 2 * kk + 1];
      const size_t o = ((tok0 + static_cast<size_t>(t) * tok_stride) * R + r) * N + 2 * kk;
      dBg[o] = cs * db0 - sn * db1;
      dBg[o + 1] = sn * db0 + cs * db1;
      dCg[o] = cs * dc0 - sn * dc1;
      dCg[o + 1] = sn * dc0 + cs * dc1;
      dph += db0 * b1 - db1 * b0 + dc0 * c1 - dc1 * c0;
    }
    sdphi[t * K + kk] = dph;
  }
  __syncthreads();
  // chunk-local suffix sums of d phi: d theta_t (this chunk's part) and their sum per pair
  for (int kk = threadIdx.x; kk < K; kk += blockDim.x) {
    float g = 0.f;
    for (int t = nt - 1; t >= 0; --t) {
      g += sdphi[t * K + kk];
      sdphi[t * K + kk] = g;
      p.dtheta[(tok0 + static_cast<size_t>(t) * tok_stride) * K + kk] = s_dt[t] * g;
    }
    p.wsSphi[(static_cast<size_t>(bh) * p.nch + k) * K + kk] = g;
  }
  __syncthreads();
  // per token: d dt (this chunk's part of the angle term), d lambda; d(dt A) by a suffix sum
  if (threadIdx.x < 32) {
    const int t = threadIdx.x;
    // d a_t = sum_{i >= t} d l_i (l_i = sum_{s <= i} a_s within the chunk)
    float da = t < nt ? s_dell[t] : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float v = __shfl_down_sync(0xffffffffu, da, o);
      if (t + o < 32) da += v;
    }
    float dadt = 0.f;
    if (t < nt) {
      float th = 0.f;
      for (int kk = 0; kk < K; ++kk) th = fmaf(s_th[t * K + kk], sdphi[t * K + kk], th);
      const float dt = s_dt[t], lam = s_lam[t];
      const size_t o = tok0 + static_cast<size_t>(t) * tok_stride;
      p.ddt[o] = th + da * A + lam * s_dgam[t] + (1.f - lam) * s_dq[t];
      p.dlam[o] = dt * (s_dgam[t] - s_dq[t]);
      dadt = da * dt;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dadt += __shfl_xor_sync(0xffffffffu, dadt, o);
    if (t == 0) p.wsDa[static_cast<size_t>(bh) * p.nch + k] = dadt;
  }
}

// ------------------------------------------------------------------ angle carries, dA part
template <typename Tin>
__global__ void __launch_bounds__(kThreads) bwd_finalize_kernel(const BwdParams p) {
  extern __shared__ float sm[];
  const int bh = blockIdx.x, b = bh / p.H, head = bh % p.H;
  const int K = p.K, c = p.c;
  float* carry = sm;  // [K] sum of d phi over the chunks after the current one
  const size_t tok_stride = p.H;
  const size_t seq0 = static_cast<size_t>(b) * p.T * p.H + head;
  const Tin* thg = static_cast<const Tin*>(p.theta);
  const Tin* dtg = static_cast<const Tin*>(p.dt);
  for (int kk = threadIdx.x; kk < K; kk += blockDim.x) carry[kk] = 0.f;
  __syncthreads();
  for (int k = p.nch - 1; k >= 0; --k) {
    const int t0 = k * c, nt = min(c, p.T - t0);
    const size_t tok0 = seq0 + static_cast<size_t>(t0) * tok_stride;
    if (k + 1 < p.nch) {
      for (int e = threadIdx.x; e < nt * K; e += blockDim.x) {
        const int t = e / K, kk = e - t * K;
        const size_t o = tok0 + static_cast<size_t>(t) * tok_stride;
        p.dtheta[o * K + kk] = fmaf(to_f(dtg[o]), carry[kk], p.dtheta[o * K + kk]);
      }
      for (int t = threadIdx.x; t < nt; t += blockDim.x) {
        const size_t o = tok0 + static_cast<size_t>(t) * tok_stride;
        float v = 0.f;
        for (int kk = 0; kk < K; ++kk) v = fmaf(to_f(thg[o * K + kk]), carry[kk], v);
        p.ddt[o] += v;
      }
    }
    __syncthreads();
    for (int kk = threadIdx.x; kk < K; kk += blockDim.x)
      carry[kk] += p.wsSphi[(static_cast<size_t>(bh) * p.nch + k) * K + kk];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int k = 0; k < p.nch; ++k) s += p.wsDa[static_cast<size_t>(bh) * p.nch + k];
    p.dApart[bh] = s;
  }
}

// dA[h] = sum over batch rows of the per-(b, h) partials, in batch order.
__global__ void dA_reduce_kernel(const float* part, float* dA, int Bsz, int H) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= H) return;
  float s = 0.f;
  for (int b = 0; b < Bsz; ++b) s += part[static_cast<size_t>(b) * H + h];
  dA[h] = s;
}

// Exit-only case (no tokens): dh0 = dhT.
__global__ void copy_dh_kernel(const float* dhT, float* dh0, size_t n) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    dh0[i] = dhT ? dhT[i] : 0.f;
}

// Tokens per chunk: the largest of 32, 16, 8, 4, 2, 1 with at most 64 (token, rank) rows whose
// per-chunk shared memory fits.
constexpr size_t kSmemLimit = 200 * 1024;
int plan_c(const m3_dims& d) {
  if (d.N * d.P > 8192) return 0;
  for (int c = kMaxTok; c >= 1; c /= 2) {
    if (c * d.R > kMaxRows) continue;
    if (static_cast<size_t>(chunk_smem(d.N, d.P, d.R, c).total) * 4 <= kSmemLimit &&
        static_cast<size_t>(scan_smem(d.N, d.P, d.R, c).total) * 4 <= kSmemLimit)
      return c;
  }
  return 0;
}

template <typename Tin, typename Tdy>
cudaError_t launch_bwd(const BackwardArgs& a, cudaStream_t s) {
  const m3_dims& d = a.d;
  const BackwardWorkspace w = backward_workspace(d);
  const size_t bhn = static_cast<size_t>(d.B) * d.H;
  cudaError_t e;
  if (d.T == 0) {
    if (a.dh0) {
      copy_dh_kernel<<<256, kThreads, 0, s>>>(a.dhT, a.dh0, bhn * d.N * d.P);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaMemsetAsync(a.dA, 0, sizeof(float) * d.H, s);
  }
  BwdParams p{};
  p.x = a.x;
  p.B = a.B;
  p.C = a.C;
  p.dt = a.dt;
  p.A = a.A;
  p.lam = a.lam;
  p.theta = a.theta;
  p.h0 = a.h0.h;
  p.phi0 = a.h0.phi;
  p.prevB0 = a.h0.prev_B;
  p.prevx0 = a.h0.prev_x;
  p.dy = a.dy;
  p.dhT = a.dhT;
  p.dx = a.dx;
  p.dB = a.dB;
  p.dC = a.dC;
  p.ddt = a.ddt;
  p.dlam = a.dlam;
  p.dtheta = a.dtheta;
  p.dh0 = a.dh0;
  p.wsPhi = reinterpret_cast<float*>(a.ws + w.off_phi);
  p.wsH = reinterpret_cast<float*>(a.ws + w.off_h);
  p.wsG = reinterpret_cast<float*>(a.ws + w.off_g);
  p.wsDH0 = reinterpret_cast<float*>(a.ws + w.off_dh0);
  p.wsSphi = reinterpret_cast<float*>(a.ws + w.off_sphi);
  p.wsDa = reinterpret_cast<float*>(a.ws + w.off_da_chunk);
  p.dApart = reinterpret_cast<float*>(a.ws + w.off_da);
  p.T = d.T;
  p.H = d.H;
  p.N = d.N;
  p.P = d.P;
  p.R = d.R;
  p.c = w.c;
  p.M = w.c * d.R;
  p.nch = w.nch;
  p.K = d.N / 2;
  const size_t sm1 = static_cast<size_t>(scan_smem(d.N, d.P, d.R, w.c).total) * 4;
  const size_t sm2 = static_cast<size_t>(chunk_smem(d.N, d.P, d.R, w.c).total) * 4;
  auto k1 = bwd_scan_kernel<Tin, Tdy>;
  auto k2 = bwd_chunk_kernel<Tin, Tdy>;
  if ((e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2)) != cudaSuccess)
    return e;
  k1<<<static_cast<unsigned>(bhn), kThreads, sm1, s>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  k2<<<static_cast<unsigned>(bhn * w.nch), kThreads, sm2, s>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bwd_finalize_kernel<Tin><<<static_cast<unsigned>(bhn), kThreads, sizeof(float) * p.K, s>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  dA_reduce_kernel<<<(d.H + 127) / 128, 128, 0, s>>>(p.dApart, a.dA, d.B, d.H);
  return cudaGetLastError();
}

}  // namespace

BackwardWorkspace backward_workspace(const m3_dims& d) {
  BackwardWorkspace w{};
  w.c = plan_c(d);
  w.nch = (w.c > 0 && d.T > 0) ? (d.T + w.c - 1) / w.c : 0;
  const size_t bh = static_cast<size_t>(d.B) * d.H, np = static_cast<size_t>(d.N) * d.P;
  const size_t K = d.N / 2, nch = w.nch;
  auto up = [](size_t v) { return (v + 255) & ~size_t(255); };
  w.off_da = 256;
  w.off_da_chunk = w.off_da + up(bh * sizeof(float));
  w.off_phi = w.off_da_chunk + up(bh * nch * sizeof(float));
  w.off_sphi = w.off_phi + up(bh * nch * K * sizeof(float));
  w.off_dh0 = w.off_sphi + up(bh * nch * K * sizeof(float));
  w.off_h = w.off_dh0 + up(bh * np * sizeof(float));
  w.off_g = w.off_h + up(bh * nch * np * sizeof(float));
  w.bytes = w.off_g + up(bh * nch * np * sizeof(float));
  return w;
}

bool backward_supported(const m3_dims& d) { return plan_c(d) > 0; }

cudaError_t launch_backward(const BackwardArgs& a, cudaStream_t s) {
  const bool bi = a.d.in_dtype == M3_BF16, bo = a.d.out_dtype == M3_BF16;
  if (bi && bo) return launch_bwd<__nv_bfloat16, __nv_bfloat16>(a, s);
  if (bi) return launch_bwd<__nv_bfloat16, float>(a, s);
  if (bo) return launch_bwd<float, __nv_bfloat16>(a, s);
  return launch_bwd<float, float>(a, s);
}

}  // namespace m3
