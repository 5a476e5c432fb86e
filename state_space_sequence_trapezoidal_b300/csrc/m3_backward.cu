// Backward pass of the prefill: gradients of y (and of the exit state h_T) with respect to
// x, B, C, dt, A, lambda, theta and the entry state h, on CUDA cores in fp32.
//
// The forward map is the recurrence of Proposition 1 with the rotation of Proposition 3 and
// the rank-R products of section 3.3 (the masked form of Eq. (7) is the same linear map), so
// its backward is the adjoint recurrence run in reverse time.  Per token t, with G the
// adjoint of h_t:
//   G += C~_t dy_t^T;  dC~_t = h_t dy_t;
//   d alpha_t = <G, h_{t-1}>;  d beta_t = <G, B~_{t-1} X_{t-1}^T>;  d gamma_t = <G, B~_t X_t^T>
//   dB~_t = gamma_t G X_t + beta_{t+1} G' X_t (carried from t + 1),  dX_t likewise with B~
//   G <- alpha_t G
// then the rotation's adjoint (dB = R(phi) dB~, d phi = sum over pairs of dB~ x dB~-rotated
// terms), the reverse cumulative sum of d phi (d theta_t = dt_t sum_{s>=t} d phi_s), and the
// chain rule through alpha = exp(dt A), beta = (1 - lambda) dt alpha, gamma = lambda dt.
//
// The reverse sweep needs h_{t-1} and h_t at every token.  One CTA per (batch row, head)
// first runs the forward recurrence and stores the state and angle every CH tokens in the
// workspace (checkpoints); the reverse sweep then recomputes each chunk of CH tokens from its
// checkpoint (states kept per thread, B~, C~, X, dy, sin/cos of the chunk in shared memory)
// and walks it backwards.  Both forward passes go a chunk at a time: the chunk's inputs are
// staged with all loads in flight, the angle and the rotation advance per pair over the chunk,
// and the state entries then run through the chunk without a barrier.  Thread (p, g) owns column p of state rows g, g + G, ...; sums over
// p go through a padded shared copy of G and h_t, sums over n through per-group partials; the
// four scalar adjoints of a token are summed by one warp in a fixed order, and dA over batch
// rows by a second kernel, so results are deterministic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "m3_internal.h"

namespace m3 {
namespace {

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

constexpr int kRows = 8;   // state rows per thread at most
constexpr int kChMax = 16; // tokens per recomputed chunk at most

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
  float* ck;      // [B*H][nch][N*P + Kp] checkpoints
  float* dApart;  // [B*H]
  int T, H, N, P, R, G, CH, nch, Kp;
};

// Shared-memory plan (floats), shared by the kernel and the host.
struct BwdSmem {
  int sB, sC, sX, sCS, sSN, sTH, sCoef, sPhi, sG, sH, sDy, redB, redBp, redA, sdB, sdC, dBn, dxn,
      partBG, gphi, partTh, total;
};

__host__ __device__ inline BwdSmem bwd_smem(int N, int P, int R, int G, int CH) {
  const int K = N / 2;
  BwdSmem s{};
  int o = 0;
  auto take = [&](int n) {
    const int at = o;
    o += (n + 3) & ~3;
    return at;
  };
  s.sB = take((CH + 1) * R * N);  // B~ of the chunk, slot 0 = the token before it
  s.sC = take(CH * R * N);        // C~
  s.sX = take((CH + 1) * R * P);  // X, slot 0 = the token before the chunk
  s.sCS = take(CH * K);
  s.sSN = take(CH * K);
  s.sTH = take(CH * K);           // theta
  s.sCoef = take(CH * 5);         // alpha, beta, gamma, dt, lambda
  s.sPhi = take(K);
  s.sG = take(N * (P + 1));       // adjoint of h_t (padded rows)
  s.sH = take(N * (P + 1));       // h_t
  s.sDy = take(CH * R * P);
  s.redB = take(G * R * P);       // per-group partial sums over n of G B~_t
  s.redBp = take(G * R * P);      // ... of G B~_{t-1}
  s.redA = take(G * P);           // ... of G h_{t-1}
  s.sdB = take(R * N);            // dB~_t
  s.sdC = take(R * N);            // dC~_t
  s.dBn = take(R * N);            // beta_{t+1} G X_t^T part of dB~_t, carried
  s.dxn = take(R * P);            // beta_{t+1} G^T B~_t part of dX_t, carried
  s.partBG = take(2 * N * R);     // d beta, d gamma partials per (n, r)
  s.gphi = take(K);               // sum_{s >= t} d phi_s
  s.partTh = take(K);
  s.total = o;
  return s;
}

__device__ __forceinline__ float wrap(float a) {
  return fmaf(-6.283185307179586f, rintf(a * 0.15915494309189535f), a);
}

// Fixed-order sum of v[0], v[stride], ..., v[(n - 1) stride] by one warp.
__device__ __forceinline__ float warp_sum(const float* v, int n, int lane, int stride = 1) {
  float s = 0.f;
  for (int i = lane; i < n; i += 32) s += v[i * stride];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

template <typename Tin, typename Tdy>
__global__ void __launch_bounds__(1024) prefill_backward_kernel(const BwdParams p) {
  const int bh = blockIdx.x;
  const int b = bh / p.H, head = bh % p.H;
  const int T = p.T, H = p.H, N = p.N, P = p.P, R = p.R, G = p.G, CH = p.CH, K = N / 2;
  const int nth = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the block is rounded up to whole warps; threads past P * G own no state entries
  const int pcol = tid % P, g = tid / P;
  const bool own = tid < P * G;
  const int rows = own ? N / G : 0;
  const BwdSmem L = bwd_smem(N, P, R, G, CH);
  extern __shared__ float sm[];
  float* sB = sm + L.sB;
  float* sC = sm + L.sC;
  float* sX = sm + L.sX;
  float* sCS = sm + L.sCS;
  float* sSN = sm + L.sSN;
  float* sTH = sm + L.sTH;
  float* sCoef = sm + L.sCoef;
  float* sPhi = sm + L.sPhi;
  float* sG = sm + L.sG;
  float* sH = sm + L.sH;
  float* sDy = sm + L.sDy;
  float* redB = sm + L.redB;
  float* redBp = sm + L.redBp;
  float* redA = sm + L.redA;
  float* sdB = sm + L.sdB;
  float* sdC = sm + L.sdC;
  float* dBn = sm + L.dBn;
  float* dxn = sm + L.dxn;
  float* partBG = sm + L.partBG;
  float* gphi = sm + L.gphi;
  float* partTh = sm + L.partTh;

  const Tin* xg = static_cast<const Tin*>(p.x);
  const Tin* Bg = static_cast<const Tin*>(p.B);
  const Tin* Cg = static_cast<const Tin*>(p.C);
  const Tin* dtg = static_cast<const Tin*>(p.dt);
  const Tin* lamg = static_cast<const Tin*>(p.lam);
  const Tin* thg = static_cast<const Tin*>(p.theta);
  const Tdy* dyg = static_cast<const Tdy*>(p.dy);
  const float A = p.A[head];
  float* ck = p.ck + static_cast<size_t>(bh) * p.nch * (static_cast<size_t>(N) * P + p.Kp);
  auto tok = [&](int t) { return (static_cast<size_t>(b) * T + t) * H + head; };  // (b, t, head)

  // Entry state and the token before t = 0 (rotated by its own angle phi0).
  float h[kRows];
#pragma unroll
  for (int i = 0; i < kRows; ++i)
    h[i] = (i < rows && p.h0) ? p.h0[(static_cast<size_t>(bh) * N + g + i * G) * P + pcol] : 0.f;
  for (int k = tid; k < K; k += nth) {
    const float ph = p.phi0 ? p.phi0[static_cast<size_t>(bh) * K + k] : 0.f;
    sPhi[k] = ph;
    float s, c;
    sincosf(ph, &s, &c);
    for (int r = 0; r < R; ++r) {
      float u = 0.f, v = 0.f;
      if (p.prevB0) {
        const Tin* pb = static_cast<const Tin*>(p.prevB0) + (static_cast<size_t>(bh) * R + r) * N;
        u = to_f(pb[2 * k]);
        v = to_f(pb[2 * k + 1]);
      }
      sB[r * N + 2 * k] = c * u + s * v;  // slot 0: the token before the first chunk
      sB[r * N + 2 * k + 1] = -s * u + c * v;
    }
  }
  for (int i = tid; i < R * P; i += nth)
    sX[i] = p.prevx0 ? to_f(static_cast<const Tin*>(p.prevx0)[static_cast<size_t>(bh) * R * P + i]) : 0.f;
  __syncthreads();

  // ------------------------------------------------------------------ forward, checkpoints
  // Chunk by chunk: the chunk's raw inputs are staged in shared memory with all loads in
  // flight together; the pair threads advance the angle and rotate B for the whole chunk; then
  // every thread runs its own state entries through the chunk with no barrier.  Slot 0 of the
  // B~ / X buffers holds the token before the chunk.
  for (int j = 0; j < p.nch; ++j) {
    const int t0 = j * CH, len = min(CH, T - t0);
    float* c0 = ck + static_cast<size_t>(j) * (static_cast<size_t>(N) * P + p.Kp);
#pragma unroll
    for (int i = 0; i < kRows; ++i)
      if (i < rows) c0[(g + i * G) * P + pcol] = h[i];
    for (int k = tid; k < K; k += nth) c0[static_cast<size_t>(N) * P + k] = sPhi[k];
    if (j > 0) {  // the previous chunk's last token moves to slot 0
      __syncthreads();
      for (int i = tid; i < R * N; i += nth) sB[i] = sB[CH * R * N + i];
      for (int i = tid; i < R * P; i += nth) sX[i] = sX[CH * R * P + i];
      __syncthreads();
    }
    for (int idx = tid; idx < len * R * N; idx += nth) {
      const int q = idx / (R * N), i = idx - q * (R * N);
      sB[(q + 1) * R * N + i] = to_f(Bg[tok(t0 + q) * R * N + i]);
    }
    for (int idx = tid; idx < len * R * P; idx += nth) {
      const int q = idx / (R * P), i = idx - q * (R * P);
      sX[(q + 1) * R * P + i] = to_f(xg[tok(t0 + q) * R * P + i]);
    }
    for (int idx = tid; idx < len * K; idx += nth) {
      const int q = idx / K, k = idx - q * K;
      sTH[q * K + k] = to_f(thg[tok(t0 + q) * K + k]);
    }
    for (int q = tid; q < len; q += nth) {
      sCoef[q * 5 + 3] = to_f(dtg[tok(t0 + q)]);
      sCoef[q * 5 + 4] = to_f(lamg[tok(t0 + q)]);
    }
    __syncthreads();
    for (int k = tid; k < K; k += nth) {
      float ph = sPhi[k];
      for (int q = 0; q < len; ++q) {
        ph = wrap(ph + sCoef[q * 5 + 3] * sTH[q * K + k]);
        float sn, cs;
        sincosf(ph, &sn, &cs);
        for (int r = 0; r < R; ++r) {
          float* bq = sB + ((q + 1) * R + r) * N + 2 * k;
          const float u = bq[0], v = bq[1];
          bq[0] = cs * u + sn * v;
          bq[1] = -sn * u + cs * v;
        }
      }
      sPhi[k] = ph;
    }
    __syncthreads();
    for (int q = 0; q < len; ++q) {
      const float dt = sCoef[q * 5 + 3], lam = sCoef[q * 5 + 4];
      const float alpha = expf(dt * A), beta = (1.f - lam) * dt * alpha, gamma = lam * dt;
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        if (i < rows) {
          const int n = g + i * G;
          float pt = 0.f, ct = 0.f;
          for (int r = 0; r < R; ++r) {
            pt = fmaf(sB[(q * R + r) * N + n], sX[(q * R + r) * P + pcol], pt);
            ct = fmaf(sB[((q + 1) * R + r) * N + n], sX[((q + 1) * R + r) * P + pcol], ct);
          }
          h[i] = fmaf(alpha, h[i], fmaf(beta, pt, gamma * ct));
        }
      }
    }
  }

  // ------------------------------------------------------------------ reverse sweep
  float Gd[kRows];
#pragma unroll
  for (int i = 0; i < kRows; ++i)
    Gd[i] = (i < rows && p.dhT) ? p.dhT[(static_cast<size_t>(bh) * N + g + i * G) * P + pcol] : 0.f;
  for (int i = tid; i < R * N; i += nth) dBn[i] = 0.f;
  for (int i = tid; i < R * P; i += nth) dxn[i] = 0.f;
  for (int k = tid; k < K; k += nth) gphi[k] = 0.f;
  float dA_acc = 0.f;
  float hs[kChMax + 1][kRows];
  __syncthreads();

  for (int j = p.nch - 1; j >= 0; --j) {
    const int t0 = j * CH, len = min(CH, T - t0);
    // recompute the chunk from its checkpoint
    const float* c0 = ck + static_cast<size_t>(j) * (static_cast<size_t>(N) * P + p.Kp);
#pragma unroll
    for (int i = 0; i < kRows; ++i) hs[0][i] = i < rows ? c0[(g + i * G) * P + pcol] : 0.f;
    for (int k = tid; k < K; k += nth) {
      const float ph = c0[static_cast<size_t>(N) * P + k];
      sPhi[k] = ph;
      float s, c;
      sincosf(ph, &s, &c);
      for (int r = 0; r < R; ++r) {
        float u = 0.f, v = 0.f;
        if (t0 > 0) {
          const size_t o = (tok(t0 - 1) * R + r) * N + 2 * k;
          u = to_f(Bg[o]);
          v = to_f(Bg[o + 1]);
        } else if (p.prevB0) {
          const Tin* pb = static_cast<const Tin*>(p.prevB0) + (static_cast<size_t>(bh) * R + r) * N;
          u = to_f(pb[2 * k]);
          v = to_f(pb[2 * k + 1]);
        }
        sB[r * N + 2 * k] = c * u + s * v;
        sB[r * N + 2 * k + 1] = -s * u + c * v;
      }
    }
    for (int i = tid; i < R * P; i += nth) {
      float v = 0.f;
      if (t0 > 0)
        v = to_f(xg[tok(t0 - 1) * R * P + i]);
      else if (p.prevx0)
        v = to_f(static_cast<const Tin*>(p.prevx0)[static_cast<size_t>(bh) * R * P + i]);
      sX[i] = v;
    }
    for (int idx = tid; idx < len * R * N; idx += nth) {
      const int q = idx / (R * N), i = idx - q * (R * N);
      sB[(q + 1) * R * N + i] = to_f(Bg[tok(t0 + q) * R * N + i]);
      sC[q * R * N + i] = to_f(Cg[tok(t0 + q) * R * N + i]);
    }
    for (int idx = tid; idx < len * R * P; idx += nth) {
      const int q = idx / (R * P), i = idx - q * (R * P);
      sX[(q + 1) * R * P + i] = to_f(xg[tok(t0 + q) * R * P + i]);
      sDy[q * R * P + i] = to_f(dyg[tok(t0 + q) * R * P + i]);
    }
    for (int idx = tid; idx < len * K; idx += nth) {
      const int q = idx / K, k = idx - q * K;
      sTH[q * K + k] = to_f(thg[tok(t0 + q) * K + k]);
    }
    for (int q = tid; q < len; q += nth) {
      const float dt = to_f(dtg[tok(t0 + q)]), lam = to_f(lamg[tok(t0 + q)]);
      const float alpha = expf(dt * A);
      sCoef[q * 5 + 0] = alpha;
      sCoef[q * 5 + 1] = (1.f - lam) * dt * alpha;
      sCoef[q * 5 + 2] = lam * dt;
      sCoef[q * 5 + 3] = dt;
      sCoef[q * 5 + 4] = lam;
    }
    __syncthreads();
    for (int k = tid; k < K; k += nth) {
      float ph = sPhi[k];
      for (int q = 0; q < len; ++q) {
        ph = wrap(ph + sCoef[q * 5 + 3] * sTH[q * K + k]);
        float sn, cs;
        sincosf(ph, &sn, &cs);
        sCS[q * K + k] = cs;
        sSN[q * K + k] = sn;
        for (int r = 0; r < R; ++r) {
          float* bq = sB + ((q + 1) * R + r) * N + 2 * k;
          float* cq = sC + (q * R + r) * N + 2 * k;
          const float bu = bq[0], bv = bq[1], cu = cq[0], cv = cq[1];
          bq[0] = cs * bu + sn * bv;
          bq[1] = -sn * bu + cs * bv;
          cq[0] = cs * cu + sn * cv;
          cq[1] = -sn * cu + cs * cv;
        }
      }
    }
    __syncthreads();
    for (int q = 0; q < len; ++q) {
      const float alpha = sCoef[q * 5 + 0], beta = sCoef[q * 5 + 1], gamma = sCoef[q * 5 + 2];
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        if (i < rows) {
          const int n = g + i * G;
          float pt = 0.f, ct = 0.f;
          for (int r = 0; r < R; ++r) {
            pt = fmaf(sB[(q * R + r) * N + n], sX[(q * R + r) * P + pcol], pt);
            ct = fmaf(sB[((q + 1) * R + r) * N + n], sX[((q + 1) * R + r) * P + pcol], ct);
          }
          hs[q + 1][i] = fmaf(alpha, hs[q][i], fmaf(beta, pt, gamma * ct));
        }
      }
    }
    __syncthreads();

    // walk the chunk backwards
    for (int q = len - 1; q >= 0; --q) {
      const int t = t0 + q;
      const float alpha = sCoef[q * 5 + 0], beta = sCoef[q * 5 + 1], gamma = sCoef[q * 5 + 2];
      const float dt = sCoef[q * 5 + 3], lam = sCoef[q * 5 + 4];
      const float* bt = sB + (q + 1) * R * N;   // B~_t
      const float* bp = sB + q * R * N;         // B~_{t-1}
      const float* ct = sC + q * R * N;         // C~_t
      const float* xt = sX + (q + 1) * R * P;   // X_t
      const float* xp = sX + q * R * P;         // X_{t-1}
      const float* dyt = sDy + q * R * P;
      // S0: G += C~_t dy_t^T; shared copies of G and h_t; partial sums over this thread's rows
      float pb[8], pbp[8], pa = 0.f;
#pragma unroll
      for (int r = 0; r < 8; ++r) pb[r] = pbp[r] = 0.f;
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        if (i < rows) {
          const int n = g + i * G;
          float gi = Gd[i];
          for (int r = 0; r < R; ++r) gi = fmaf(ct[r * N + n], dyt[r * P + pcol], gi);
          Gd[i] = gi;
          sG[n * (P + 1) + pcol] = gi;
          sH[n * (P + 1) + pcol] = hs[q + 1][i];
          pa = fmaf(gi, hs[q][i], pa);
#pragma unroll
          for (int r = 0; r < 8; ++r)
            if (r < R) {
              pb[r] = fmaf(gi, bt[r * N + n], pb[r]);
              pbp[r] = fmaf(gi, bp[r * N + n], pbp[r]);
            }
          Gd[i] = alpha * gi;  // adjoint of h_{t-1}
        }
      }
      if (own) {
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (r < R) {
            redB[(g * R + r) * P + pcol] = pb[r];
            redBp[(g * R + r) * P + pcol] = pbp[r];
          }
        redA[g * P + pcol] = pa;
      }
      __syncthreads();
      // S1: sums over p (per (n, r), eight lanes per (n, r) and a fixed shuffle tree; the loop
      // runs over whole warps so that every lane takes part in the shuffles) and over n (per (p, r))
      for (int t8 = tid; t8 < (N * R * 8 + 31) / 32 * 32; t8 += nth) {
        const int task = t8 >> 3, sub = t8 & 7;
        const bool valid = task < N * R;
        const int n = valid ? task / R : 0, r = valid ? task - n * R : 0;
        float dc = 0.f, gx = 0.f, gxp = 0.f;
        if (valid) {
          const float* grow = sG + n * (P + 1);
          const float* hrow = sH + n * (P + 1);
          for (int pp = sub; pp < P; pp += 8) {
            dc = fmaf(hrow[pp], dyt[r * P + pp], dc);
            gx = fmaf(grow[pp], xt[r * P + pp], gx);
            gxp = fmaf(grow[pp], xp[r * P + pp], gxp);
          }
        }
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) {
          dc += __shfl_xor_sync(0xffffffffu, dc, o);
          gx += __shfl_xor_sync(0xffffffffu, gx, o);
          gxp += __shfl_xor_sync(0xffffffffu, gxp, o);
        }
        if (valid && sub == 0) {
          sdC[r * N + n] = dc;
          sdB[r * N + n] = fmaf(gamma, gx, dBn[r * N + n]);
          dBn[r * N + n] = beta * gxp;
          partBG[2 * task] = bp[r * N + n] * gxp;      // d beta
          partBG[2 * task + 1] = bt[r * N + n] * gx;   // d gamma
        }
      }
      for (int task = tid; task < P * R; task += nth) {
        const int r = task / P, pp = task - r * P;
        float gb = 0.f, gbp = 0.f;
        for (int gg = 0; gg < G; ++gg) {
          gb += redB[(gg * R + r) * P + pp];
          gbp += redBp[(gg * R + r) * P + pp];
        }
        const size_t o = tok(t) * R * P + static_cast<size_t>(r) * P + pp;
        p.dx[o] = fmaf(gamma, gb, dxn[r * P + pp]);
        dxn[r * P + pp] = beta * gbp;
      }
      __syncthreads();
      // S2: the rotation's adjoint, pair by pair
      for (int k = tid; k < K; k += nth) {
        const float c = sCS[q * K + k], s = sSN[q * K + k];
        float dphi = 0.f;
        for (int r = 0; r < R; ++r) {
          const float b0 = bt[r * N + 2 * k], b1 = bt[r * N + 2 * k + 1];
          const float c0 = ct[r * N + 2 * k], c1 = ct[r * N + 2 * k + 1];
          const float db0 = sdB[r * N + 2 * k], db1 = sdB[r * N + 2 * k + 1];
          const float dc0 = sdC[r * N + 2 * k], dc1 = sdC[r * N + 2 * k + 1];
          dphi += db0 * b1 - db1 * b0 + dc0 * c1 - dc1 * c0;
          const size_t o = (tok(t) * R + r) * N + 2 * k;
          p.dB[o] = c * db0 - s * db1;
          p.dB[o + 1] = s * db0 + c * db1;
          p.dC[o] = c * dc0 - s * dc1;
          p.dC[o + 1] = s * dc0 + c * dc1;
        }
        const float gk = gphi[k] + dphi;
        gphi[k] = gk;
        p.dtheta[tok(t) * K + k] = dt * gk;
        partTh[k] = sTH[q * K + k] * gk;
      }
      __syncthreads();
      // S3: the token's scalar adjoints (one warp, fixed order)
      if (warp == 0) {
        const float da = warp_sum(redA, G * P, lane);
        const float db = warp_sum(partBG, N * R, lane, 2);
        const float dg = warp_sum(partBG + 1, N * R, lane, 2);
        const float dph = warp_sum(partTh, K, lane);
        if (lane == 0) {
          p.ddt[tok(t)] = da * alpha * A + db * (1.f - lam) * alpha * fmaf(dt, A, 1.f) + dg * lam + dph;
          p.dlam[tok(t)] = dt * (dg - alpha * db);
          dA_acc += (da * alpha + db * (1.f - lam) * dt * alpha) * dt;
        }
      }
      __syncthreads();
    }
  }

  // ------------------------------------------------------------------ entry-state outputs
  if (p.dh0) {
#pragma unroll
    for (int i = 0; i < kRows; ++i)
      if (i < rows) p.dh0[(static_cast<size_t>(bh) * N + g + i * G) * P + pcol] = Gd[i];
  }
  if (tid == 0) p.dApart[bh] = dA_acc;
}

// dA[h] = sum over batch rows of the per-(b, h) partials, in batch order.
__global__ void dA_reduce_kernel(const float* part, float* dA, int Bsz, int H) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= H) return;
  float s = 0.f;
  for (int b = 0; b < Bsz; ++b) s += part[static_cast<size_t>(b) * H + h];
  dA[h] = s;
}

// Row groups: the smallest G >= ceil(N / kRows) dividing N, with P * G threads (rounded up
// to whole warps) <= 1024.
int plan_g(const m3_dims& d) {
  for (int g = (d.N + kRows - 1) / kRows; g <= d.N; ++g)
    if (d.N % g == 0) return (d.P * g + 31) / 32 * 32 <= 1024 ? g : 0;
  return 0;
}

// Tokens per recomputed chunk: the largest of 16, 8, 4, 2 whose shared memory fits.
int plan_ch(const m3_dims& d, int G) {
  for (int ch = kChMax; ch >= 2; ch /= 2)
    if (static_cast<size_t>(bwd_smem(d.N, d.P, d.R, G, ch).total) * 4 <= 200 * 1024) return ch;
  return 0;
}

template <typename Tin, typename Tdy>
cudaError_t launch_bwd(const BackwardArgs& a, cudaStream_t s) {
  const m3_dims& d = a.d;
  const int G = plan_g(d), CH = plan_ch(d, G);
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
  const BackwardWorkspace w = backward_workspace(d);
  p.ck = reinterpret_cast<float*>(a.ws + w.off_ck);
  p.dApart = reinterpret_cast<float*>(a.ws + w.off_da);
  p.T = d.T;
  p.H = d.H;
  p.N = d.N;
  p.P = d.P;
  p.R = d.R;
  p.G = G;
  p.CH = CH;
  p.nch = w.nch;
  p.Kp = w.kp;
  const size_t smem = static_cast<size_t>(bwd_smem(d.N, d.P, d.R, G, CH).total) * 4;
  auto k = prefill_backward_kernel<Tin, Tdy>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int threads = (d.P * G + 31) / 32 * 32;
  k<<<static_cast<unsigned>(d.B) * static_cast<unsigned>(d.H), threads, smem, s>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  dA_reduce_kernel<<<(d.H + 127) / 128, 128, 0, s>>>(p.dApart, a.dA, d.B, d.H);
  return cudaGetLastError();
}

}  // namespace

BackwardWorkspace backward_workspace(const m3_dims& d) {
  BackwardWorkspace w{};
  w.nch = 0;
  w.kp = ((d.N / 2) + 3) & ~3;
  const int G = plan_g(d);
  const int CH = G ? plan_ch(d, G) : 0;
  if (CH > 0 && d.T > 0) w.nch = (d.T + CH - 1) / CH;
  const size_t bh = static_cast<size_t>(d.B) * d.H;
  auto up = [](size_t v) { return (v + 255) & ~size_t(255); };
  w.off_da = 256;
  w.off_ck = w.off_da + up(bh * sizeof(float));
  w.bytes = w.off_ck + up(bh * w.nch * (static_cast<size_t>(d.N) * d.P + w.kp) * sizeof(float));
  return w;
}

bool backward_supported(const m3_dims& d) {
  const int G = plan_g(d);
  return G > 0 && plan_ch(d, G) > 0;
}

cudaError_t launch_backward(const BackwardArgs& a, cudaStream_t s) {
  const bool bi = a.d.in_dtype == M3_BF16, bo = a.d.out_dtype == M3_BF16;
  if (bi && bo) return launch_bwd<__nv_bfloat16, __nv_bfloat16>(a, s);
  if (bi) return launch_bwd<__nv_bfloat16, float>(a, s);
  if (bo) return launch_bwd<float, __nv_bfloat16>(a, s);
  return launch_bwd<float, float>(a, s);
}

}  // namespace m3
