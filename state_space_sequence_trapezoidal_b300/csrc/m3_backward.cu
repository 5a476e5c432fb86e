// Backward pass of the prefill: gradients of y (and of the exit state h_T) with respect to
// x, B, C, dt, A, lambda, theta and the entry state h, in fp32 (the chunk products on the
// tensor cores as three TF32 passes, the rest on CUDA cores).
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
//   dB~_s = sum_i D[i, s]^T C~_i + wx_s X_s Gout^T
//   dX_s  = sum_i Mh[i, s] (C~_i B~_s^T)^T dY_i + wx_s B~_s Gout
//   dHp   = exp(l_last) Gout + sum_i exp(l_i) C~_i^T dY_i
//   dMh[i, s] = <C~_i B~_s^T, dY_i X_s^T> (+ <Gout, B~_s^T X_s> on the last row)
// where wx_s = Mh[last, s], plus q of the next chunk's first token for the last token (its
// trapezoid term is folded into the next chunk's Hp).  Then the chain rule through l, w,
// gamma, q, the fold and the rotation (dB = R(phi) dB~, d phi from the rotation's
// derivative, d theta_t = dt_t sum_{s>=t} d phi_s over the whole sequence).  MIMO rank R:
// rows are (token, rank) pairs and every rank pair of two tokens shares their mask entry.
//
// Frames.  Every chunk works in its own frame: B~, C~ rotated by the angle accumulated from
// the chunk's start (psi_t), not from the sequence's.  Since the rotations of one pair
// commute, the absolute B~ is the local one turned by the angle phi_b before the chunk, and a
// state Z (rows = state entries) reads Z_loc = R(-phi_b) Z in the chunk's frame; inner products
// over the state entries are the same in either frame.  Going from chunk k to k + 1 turns a
// state by the chunk's angle advance sigma_k = psi_last.  Only the entry state (angle phi_0)
// and the exit cotangent (angle before the last chunk) meet absolute angles.
//
// Kernels, in launch order:
//   bwd_local_kernel   one CTA per (batch row, head, chunk): the chunk's own contributions to
//                      the next chunk's folded state, dH = sum_s wx_s B~_s^T X_s, and to the
//                      previous chunk's exit cotangent, dG = sum_i exp(l_i) C~_i^T dY_i (both
//                      local frame), exp(l_last) and sigma.
//   bwd_scan_kernel    one thread per (batch row, head, state pair, column), forward (Hp) or
//                      reverse (Gout) over the chunks: Hp(k+1) = R(-sigma_k)(exp(l_last) Hp(k)
//                      + dH(k)), Gout(k-1) = R(sigma_{k-1})(exp(l_last) Gout(k) + dG(k)), each
//                      written over its chunk's dH / dG.
//   bwd_chunk_kernel   persistent, one CTA per SM walking chunks (batch row, head, chunk): the
//                      adjoint above, the mask and fold parameters, the rotation adjoint,
//                      chunk-local suffix sums of d phi; the next chunk's theta, Hp, Gout and
//                      coefficients are requested while the current one finishes.
//   bwd_carry_kernel   one CTA per (batch row, head): suffix sums of d phi over chunks, the
//                      per-(b, h) part of dA, the fold gradient of the sequence's first token.
//   bwd_apply_kernel   one CTA per (batch row, head, chunk): adds the later chunks' d phi to
//                      d theta and d dt, and the fold gradient of the chunk's first token.
//   dA_reduce_kernel   sums dA over batch rows.
// Every reduction has a fixed order, so results are bit-identical from run to run.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include <cudaTypedefs.h>

#include "m3_internal.h"
#include "m3_ptx.cuh"

namespace m3 {
namespace {

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

constexpr int kThreads = 256;       // threads of the local, carry and apply kernels
constexpr int kThreadsChunk = 512;  // threads of the adjoint kernel
constexpr int kPad = 4;        // floats of padding at the end of each shared-memory row
constexpr int kPadT = 8;       // the same for rows read only across (the local kernel's inputs)
constexpr int kMaxRows = 64;   // (token, rank) rows per chunk at most
constexpr int kMaxTok = 32;    // tokens per chunk at most (one warp lane each)

struct BwdParams {
  CUtensorMap tmH;  // wsH as [BH nch N][P] fp32, box {32, N}, 128-byte swizzle (swizzled states only)
  CUtensorMap tmG;  // wsG, the same
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
  float* wsH;     // [BH][nch][N*P]  dH(k), then Hp(k) (chunk k's frame)
  float* wsG;     // [BH][nch][N*P]  dG(k), then Gout(k) (chunk k's frame)
  float* wsSig;   // [BH][nch][K]    angle advance over chunk k, reduced to [-pi, pi]
  float* wsDec;   // [BH][nch]       exp(l_last) of chunk k
  float* wsDH0;   // [BH][N*P]       cotangent of Hp(0) in chunk 0's frame
  float* wsSphi;  // [BH][nch][K]    sum of d phi over chunk k, then over the chunks after k
  float* wsDa;    // [BH][nch]       sum over chunk k's tokens of d(dt A) * dt
  float* wsDqf;   // [BH][nch]       d q of chunk k's first token through the fold
  float* dApart;  // [BH]
  unsigned* status;  // device status word (a bounded wait that ran out: kDevTimeout)
  int T, H, N, P, R, c, M, nch, K;
  int BH;  // sequences (batch rows x heads)
};

__device__ __forceinline__ float wrap(float a) {
  return fmaf(-6.283185307179586f, rintf(a * 0.15915494309189535f), a);
}

// The chunk geometry.  Kernels specialised for a shape take compile-time values, which the
// inlined helpers below fold into their index arithmetic; 0 means "from the parameters".
struct Shape {
  int N, P, R, c, K, M;
};
template <int SN, int SP, int SR, int SC>
__device__ __forceinline__ Shape shape_of(const BwdParams& p) {
  Shape s;
  s.N = SN ? SN : p.N;
  s.P = SP ? SP : p.P;
  s.R = SR ? SR : p.R;
  s.c = SC ? SC : p.c;
  s.K = s.N / 2;
  s.M = s.c * s.R;
  return s;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(
                   __cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// A {32 columns, rows} box of a 2-D fp32 tensor map into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
// Float offset of state entry (n, p) in a state of `rows` rows stored by tma_load_2d with the
// 128-byte swizzle: 32-column boxes of rows x 128 B, the 16-byte group of p within its 128-byte
// row turned by n mod 8 (the destination is 1024-byte aligned).
__device__ __forceinline__ int swz(int n, int p, int rows) {
  return (p >> 5) * (rows * 32) + n * 32 + ((((p & 31) >> 2) ^ (n & 7)) << 2) + (p & 3);
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Register-tiled product on the CUDA cores, for the shapes the tensor-core product below does
// not take: out(i, j, sum_k A(i, k) B(k, j)) for i < NI, j < NJ, with A(i, k) = a[i * lda + k]
// when kAK (k contiguous), else a[k * lda + i], and B(k, j) = b[j * ldb + k] when kBK, else
// b[k * ldb + j].  A warp computes a (4 TI) x (8 TJ) tile; lane (gi, gj) = (lane / 8, lane % 8)
// owns rows gi + 4 u and columns gj + 8 v of it, so that the rows one load instruction touches
// fall in distinct banks for row strides of 4 (mod 32) words.  Reads past NI / NJ are clamped
// to valid rows / columns and their results dropped.  Warp tiles continue the round-robin of
// the previous product through rr, so that products issued back to back without a barrier
// share the warps evenly.
template <int TI, int TJ, bool kAK, bool kBK, typename FO>
__device__ __forceinline__ void gemm(int& rr, int NI, int NJ, int NK, const float* __restrict__ a,
                                     int lda, const float* __restrict__ b, int ldb, FO out) {
  constexpr int WI = 4 * TI, WJ = 8 * TJ;
  const int lane = threadIdx.x & 31, nw = static_cast<int>(blockDim.x >> 5);
  const int gi = lane >> 3, gj = lane & 7;
  const int nwj = (NJ + WJ - 1) / WJ, ntile = ((NI + WI - 1) / WI) * nwj;
  int w = static_cast<int>(threadIdx.x >> 5) - rr % nw;
  if (w < 0) w += nw;
  rr += ntile;
  for (int t = w; t < ntile; t += nw) {
    const int wi = (t / nwj) * WI, wj = (t % nwj) * WJ;
    int ri[TI], rc[TI], cj[TJ], cc[TJ];
#pragma unroll
    for (int u = 0; u < TI; ++u) {
      ri[u] = wi + gi + 4 * u;
      rc[u] = min(ri[u], NI - 1);
    }
#pragma unroll
    for (int v = 0; v < TJ; ++v) {
      cj[v] = wj + gj + 8 * v;
      cc[v] = min(cj[v], NJ - 1);
    }
    float acc[TI][TJ];
#pragma unroll
    for (int u = 0; u < TI; ++u)
#pragma unroll
      for (int v = 0; v < TJ; ++v) acc[u][v] = 0.f;
#pragma unroll 2
    for (int k = 0; k < NK; ++k) {
      float av[TI], bv[TJ];
#pragma unroll
      for (int u = 0; u < TI; ++u) av[u] = kAK ? a[rc[u] * lda + k] : a[k * lda + rc[u]];
#pragma unroll
      for (int v = 0; v < TJ; ++v) bv[v] = kBK ? b[cc[v] * ldb + k] : b[k * ldb + cc[v]];
#pragma unroll
      for (int u = 0; u < TI; ++u)
#pragma unroll
        for (int v = 0; v < TJ; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
    }
#pragma unroll
    for (int u = 0; u < TI; ++u)
#pragma unroll
      for (int v = 0; v < TJ; ++v)
        if (ri[u] < NI && cj[v] < NJ) out(ri[u], cj[v], acc[u][v]);
  }
}

// ------------------------------------------------------------------ tensor-core products
// fp32 values as TF32 pairs: x = hi + lo with hi = x rounded to TF32's 10 mantissa bits (round
// half away from zero, by integer adds and masks on the ALU rather than a conversion
// instruction) and lo = x - hi, exact in fp32, of which the MMA reads the top 19 bits (TF32)
// of its register.  A product taken as a_lo b_hi + a_hi b_lo + a_hi b_hi (the lo lo term
// dropped) keeps about 21 bits of each operand, the accuracy of an fp32 dot product here.
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = (__float_as_uint(x) + 0x1000u) & 0xffffe000u;
  lo = __float_as_uint(x - __uint_as_float(hi));
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// The product of gemm() on the tensor cores: warp-level m16n8k8 TF32 MMAs in three passes per
// fragment pair (split_tf32), summed over k in fp32 registers.  A warp computes a (16 MI) x
// (8 NJ) tile; fragments are read from shared memory with 32-bit loads in the MMA's register
// layout (lane = 4 g + t: A rows g, g + 8, k t, t + 4; B k t, t + 4, column g; D rows g, g + 8,
// columns 2 t, 2 t + 1).  With row strides of 4 (mod 32) words the loads along a k-contiguous
// operand are free of bank conflicts (4 g + t); along an index-contiguous one two lanes share
// a bank.  Needs NI % 16 == 0, NJ % 8 == 0 and NK % 8 == 0 (fragments wholly in or out); the
// in / out tests are the same for all lanes of a warp, as mma.sync requires.
template <int MI, int NJ, bool kAK, bool kBK, bool kSwzB, typename FO>
__device__ __forceinline__ void gemm_tc(int& rr, int NI, int NJd, int NK, const float* __restrict__ a,
                                        int lda, const float* __restrict__ b, int ldb, FO out) {
  constexpr int WI = 16 * MI, WJ = 8 * NJ;
  const int lane = threadIdx.x & 31, nw = static_cast<int>(blockDim.x >> 5);
  const int g = lane >> 2, t = lane & 3;
  const int nwj = (NJd + WJ - 1) / WJ, ntile = ((NI + WI - 1) / WI) * nwj;
  int w = static_cast<int>(threadIdx.x >> 5) - rr % nw;
  if (w < 0) w += nw;
  rr += ntile;
  auto A = [&](int i, int k) { return kAK ? a[i * lda + k] : a[k * lda + i]; };
  // kSwzB: b is a state in the swizzled layout of swz() with ldb rows; B(k, j) = state(j, k) when
  // kBK, else state(k, j)
  auto B = [&](int k, int j) {
    if constexpr (kSwzB)
      return kBK ? b[swz(j, k, ldb)] : b[swz(k, j, ldb)];
    else
      return kBK ? b[j * ldb + k] : b[k * ldb + j];
  };
  for (int tile = w; tile < ntile; tile += nw) {
    const int i0 = (tile / nwj) * WI, j0 = (tile % nwj) * WJ;
    float acc[MI][NJ][4];
#pragma unroll
    for (int mi = 0; mi < MI; ++mi)
#pragma unroll
      for (int nj = 0; nj < NJ; ++nj) acc[mi][nj][0] = acc[mi][nj][1] = acc[mi][nj][2] = acc[mi][nj][3] = 0.f;
#pragma unroll 2
    for (int k0 = 0; k0 < NK; k0 += 8) {
      uint32_t ah[MI][4], al[MI][4], bh[NJ][2], bl[NJ][2];
#pragma unroll
      for (int mi = 0; mi < MI; ++mi) {
        if (i0 + 16 * mi < NI) {
          const int r0 = i0 + 16 * mi + g;
          split_tf32(A(r0, k0 + t), ah[mi][0], al[mi][0]);
          split_tf32(A(r0 + 8, k0 + t), ah[mi][1], al[mi][1]);
          split_tf32(A(r0, k0 + t + 4), ah[mi][2], al[mi][2]);
          split_tf32(A(r0 + 8, k0 + t + 4), ah[mi][3], al[mi][3]);
        }
      }
#pragma unroll
      for (int nj = 0; nj < NJ; ++nj) {
        if (j0 + 8 * nj < NJd) {
          const int c = j0 + 8 * nj + g;
          split_tf32(B(k0 + t, c), bh[nj][0], bl[nj][0]);
          split_tf32(B(k0 + t + 4, c), bh[nj][1], bl[nj][1]);
        }
      }
      // each k-step's three passes into a fresh accumulator, added to the running sums by fp32
      // adds: chained along k inside the MMA the sums drift low (measured on the MIMO
      // rank-4 backward at T 4096: d theta 2.5e-4 of its RMS chained, 7.7e-5 this way, 8.2e-5
      // with the CUDA-core product)
#pragma unroll
      for (int mi = 0; mi < MI; ++mi)
#pragma unroll
        for (int nj = 0; nj < NJ; ++nj)
          if (i0 + 16 * mi < NI && j0 + 8 * nj < NJd) {
            float part[4] = {0.f, 0.f, 0.f, 0.f};
            mma_tf32(part, al[mi], bh[nj]);
            mma_tf32(part, ah[mi], bl[nj]);
            mma_tf32(part, ah[mi], bh[nj]);
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[mi][nj][r] += part[r];
          }
    }
#pragma unroll
    for (int mi = 0; mi < MI; ++mi)
#pragma unroll
      for (int nj = 0; nj < NJ; ++nj)
        if (i0 + 16 * mi < NI && j0 + 8 * nj < NJd) {
          const int r0 = i0 + 16 * mi + g, c0 = j0 + 8 * nj + 2 * t;
          out(r0, c0, acc[mi][nj][0]);
          out(r0, c0 + 1, acc[mi][nj][1]);
          out(r0 + 8, c0, acc[mi][nj][2]);
          out(r0 + 8, c0 + 1, acc[mi][nj][3]);
        }
  }
}

// The product on the tensor cores where the shapes allow (kV: N % 16, P % 8 and the row count
// M % 16 all zero, operands 16-byte aligned), else on the CUDA cores.
template <int MI, int NJ, int TI, int TJ, bool kAK, bool kBK, bool kV, typename FO>
__device__ __forceinline__ void product(int& rr, int NI, int NJd, int NK, const float* __restrict__ a,
                                        int lda, const float* __restrict__ b, int ldb, FO out) {
  if constexpr (kV)
    gemm_tc<MI, NJ, kAK, kBK, false>(rr, NI, NJd, NK, a, lda, b, ldb, out);
  else
    gemm<TI, TJ, kAK, kBK>(rr, NI, NJd, NK, a, lda, b, ldb, out);
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

// ------------------------------------------------------------------ shared-memory plans
struct Carve {
  int o = 0;
  __host__ __device__ int take(int n) {
    const int at = o;
    o += (n + 3) & ~3;
    return at;
  }
};
// floats of staging for M x len elements of sz bytes copied raw (none for fp32: copied in place)
__host__ __device__ inline int raw_floats(int M, int len, int sz) {
  return sz == 4 ? 0 : (M * len * sz + 3) / 4;
}

// Per-chunk inputs shared by the local and adjoint kernels.
struct InSmem {
  int ldN, ldP;                    // row strides of the fp32 rows: N + pad, P + pad
  int Bt, Ct, X, dY;               // fp32 rows [M][ldN] / [M][ldP]
  int rB, rC, rX, rY;              // raw staging of 16-bit inputs
  int th, cs, sn;                  // theta as loaded, cos / sin of psi [c][K]
  int dt, lam, ell, el, gam, q;    // per token (q: c + 1, the next chunk's first token last)
  int wx, rowel;                   // per row
  int part;                        // scratch of the angle pass
};
__host__ __device__ inline void carve_inputs(Carve& cv, InSmem& s, int N, int P, int R, int c, int szIn,
                                             int szDy, int raw_at, int pad, bool theta_here = true) {
  const int K = N / 2, M = c * R;
  s.ldN = N + pad;
  s.ldP = P + pad;
  s.Bt = cv.take(M * s.ldN);
  s.Ct = cv.take(M * s.ldN);
  s.X = cv.take(M * s.ldP);
  s.dY = cv.take(M * s.ldP);
  s.th = theta_here ? cv.take((c * K * szIn + 3) / 4) : -1;
  s.cs = cv.take(c * K);
  s.sn = cv.take(c * K);
  s.dt = cv.take(c);
  s.lam = cv.take(c);
  s.ell = cv.take(c);
  s.el = cv.take(c);
  s.gam = cv.take(c);
  s.q = cv.take(c + 1);
  s.wx = cv.take(M);
  s.rowel = cv.take(M);
  s.part = cv.take(K > kThreadsChunk ? K : kThreadsChunk);
  // raw staging: at raw_at when given (an area free until the inputs are converted)
  Carve rc;
  rc.o = raw_at >= 0 ? raw_at : cv.o;
  s.rB = rc.take(raw_floats(M, N, szIn));
  s.rC = rc.take(raw_floats(M, N, szIn));
  s.rX = rc.take(raw_floats(M, P, szIn));
  s.rY = rc.take(raw_floats(M, P, szDy));
  if (raw_at < 0) cv.o = rc.o;
}
__host__ __device__ inline int raw_total(int N, int P, int R, int c, int szIn, int szDy) {
  const int M = c * R;
  auto r4 = [](int n) { return (n + 3) & ~3; };
  return r4(raw_floats(M, N, szIn)) * 2 + r4(raw_floats(M, P, szIn)) + r4(raw_floats(M, P, szDy));
}

struct LocalSmem {
  InSmem in;
  int total;
};
__host__ __device__ inline LocalSmem local_smem(int N, int P, int R, int c, int szIn, int szDy) {
  LocalSmem s{};
  Carve cv;
  carve_inputs(cv, s.in, N, P, R, c, szIn, szDy, -1, kPadT);
  s.total = cv.o;
  return s;
}

struct ChunkSmem {
  InSmem in;
  int Q, XG, W, Hp, Go, S, E, th, dphi, Mh, ex, dM, dexp, wdot, dell, dgam, dq, red, bar, total;
};
// swz_state: Hp and Gout dense in the swizzled layout of swz(), each at a 1024-byte boundary of
// a base that the kernel aligns to 1024 bytes; else rows padded to P + kPad.
__host__ __device__ inline ChunkSmem chunk_smem(int N, int P, int R, int c, int szIn, int szDy,
                                                bool swz_state = false) {
  const int K = N / 2, M = c * R;
  ChunkSmem s{};
  Carve cv;
  s.Q = cv.take(M * (N + kPad));   // dY Hp^T, then dC~
  s.XG = cv.take(M * (N + kPad));  // X Gout^T, then dB~
  // the raw inputs wait in Q and XG when they fit there (both are written after conversion)
  const int raw = raw_total(N, P, R, c, szIn, szDy);
  carve_inputs(cv, s.in, N, P, R, c, szIn, szDy, raw <= 2 * M * (N + kPad) ? s.Q : -1, kPad, false);
  s.W = cv.take(M * (P + kPad));   // B~ Gout; then d phi per (token, pair), where it fits
  if (swz_state) cv.o = (cv.o + 255) & ~255;
  s.Hp = cv.take(N * (swz_state ? P : P + kPad));  // Hp; the next chunk's from the end of the first products
  s.Go = cv.take(N * (swz_state ? P : P + kPad));  // Gout, likewise
  s.S = cv.take(M * (M + kPad));   // C~ B~^T, then Mh o S; then the next chunk's theta
  s.E = cv.take(M * (M + kPad));   // dY X^T, then Mh o E
  s.th = c * K <= 2 * M * (M + kPad) ? s.S : cv.take(c * K);  // theta, fp32 or raw 16-bit
  s.dphi = c * K <= M * (P + kPad) ? s.W : cv.take(c * K);
  s.Mh = cv.take(c * (c + 1));
  s.ex = cv.take(c * (c + 1));
  s.dM = cv.take(c * (c + 1));
  s.dexp = cv.take(c);
  s.wdot = cv.take(c);
  s.dell = cv.take(c);
  s.dgam = cv.take(c);
  s.dq = cv.take(c);
  s.red = cv.take(kThreadsChunk);
  s.bar = cv.take(4);  // mbarrier of the swizzled state copies
  s.total = cv.o;
  return s;
}

// ------------------------------------------------------------------ chunk inputs
struct ChunkPos {
  int k, t0, nt, last;
  bool has_next;
  size_t tok0;  // index of (b, t0, h) in [B][T][H]
};
__device__ __forceinline__ ChunkPos chunk_pos(const BwdParams& p, int bh, int k, int c) {
  ChunkPos q;
  const int b = bh / p.H, head = bh % p.H;
  q.k = k;
  q.t0 = k * c;
  q.nt = min(c, p.T - q.t0);
  q.last = q.nt - 1;
  q.has_next = k + 1 < p.nch;
  q.tok0 = (static_cast<size_t>(b) * p.T + q.t0) * p.H + head;
  return q;
}

// Rows (token t < c, rank r) of a [T][H][R][len] operand of the chunk into dst[M][ld] as fp32,
// rows of tokens >= nt zero.  kV: 16-byte asynchronous copies, straight into dst for fp32 or
// into raw for 16-bit types (converted by finish_rows); else plain scalar loads.
template <typename T, bool kV>
__device__ __forceinline__ void issue_rows(const T* src, const ChunkPos& q, size_t tok_stride, int c, int R, int len,
                           float* dst, int ld, T* raw) {
  if constexpr (kV) {
    constexpr int vec = 16 / sizeof(T);
    const int per_row = len / vec, n = c * R * per_row;
    for (int e = threadIdx.x; e < n; e += blockDim.x) {
      const int row = e / per_row, col = (e - row * per_row) * vec, t = row / R;
      if (t < q.nt) {
        const T* g = src + ((q.tok0 + static_cast<size_t>(t) * tok_stride) * R + (row - t * R)) * len + col;
        if constexpr (sizeof(T) == 4)
          cp_async16(dst + row * ld + col, g);
        else
          cp_async16(raw + row * len + col, g);
      } else if constexpr (sizeof(T) == 4) {
        *reinterpret_cast<float4*>(dst + row * ld + col) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  } else {
    const int n = c * R * len;
    for (int base = threadIdx.x; base < n; base += 4 * blockDim.x) {
      float v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = base + u * blockDim.x, row = e / len, t = row / R;
        v[u] = e < n && t < q.nt
                   ? to_f(src[((q.tok0 + static_cast<size_t>(t) * tok_stride) * R + (row - t * R)) * len + (e - row * len)])
                   : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = base + u * blockDim.x, row = e / len;
        if (e < n) dst[row * ld + (e - row * len)] = v[u];
      }
    }
  }
}

// After the copies have landed: each row's values (raw 16-bit staging, or dst in place),
// rotated pairwise by the token's psi when rot, times rowscale[row] when given, into dst.
template <typename T, bool kV>
__device__ __forceinline__ void finish_rows(const ChunkPos& q, int c, int R, int len, float* dst, int ld, const T* raw,
                            bool rot, const float* s_cs, const float* s_sn, int K, const float* rowscale) {
  constexpr bool kRaw = kV && sizeof(T) != 4;
  const int M = c * R;
  if (rot) {
    for (int e = threadIdx.x; e < M * K; e += blockDim.x) {
      const int row = e / K, kk = e - row * K, t = row / R;
      float o0 = 0.f, o1 = 0.f;  // rows past nt: zero (their raw staging was never written)
      if (t < q.nt) {
        float u, v;
        if constexpr (kRaw) {
          u = to_f(raw[row * len + 2 * kk]);
          v = to_f(raw[row * len + 2 * kk + 1]);
        } else {
          u = dst[row * ld + 2 * kk];
          v = dst[row * ld + 2 * kk + 1];
        }
        const float cs = s_cs[t * K + kk], sn = s_sn[t * K + kk];
        const float sc = rowscale ? rowscale[row] : 1.f;
        o0 = sc * fmaf(cs, u, sn * v);
        o1 = sc * fmaf(cs, v, -sn * u);
      }
      dst[row * ld + 2 * kk] = o0;
      dst[row * ld + 2 * kk + 1] = o1;
    }
  } else if (kRaw || rowscale) {
    for (int e = threadIdx.x; e < M * len; e += blockDim.x) {
      const int row = e / len, col = e - row * len, t = row / R;
      float o = 0.f;
      if (t < q.nt) {
        const float u = kRaw ? to_f(raw[e]) : dst[row * ld + col];
        o = rowscale ? rowscale[row] * u : u;
      }
      dst[row * ld + col] = o;
    }
  }
}

// Per-token coefficients (warp 0, one lane per token, tokens >= nt zero): dt, lambda, the
// chunk-local log-decay sums l, exp(l), gamma, q, and q of the next chunk's first token.
// dt and lambda of the chunk's tokens (lane t of warp 0; zero past nt), of the next chunk's first
// token (lane 0), and the head's A (warp 0), for chunk_coefs.
struct CoefIn {
  float dt, lam, dtn, lamn, A;
};
template <typename Tin>
__device__ __forceinline__ CoefIn load_coefs(const BwdParams& p, const ChunkPos& q) {
  CoefIn v{0.f, 0.f, 0.f, 0.f, 0.f};
  if (threadIdx.x < 32) {
    v.A = p.A[(q.tok0 % p.H)];
    const Tin* dtg = static_cast<const Tin*>(p.dt);
    const Tin* lamg = static_cast<const Tin*>(p.lam);
    const int t = threadIdx.x;
    if (t < q.nt) {
      const size_t o = q.tok0 + static_cast<size_t>(t) * p.H;
      v.dt = to_f(dtg[o]);
      v.lam = to_f(lamg[o]);
    }
    if (t == 0 && q.has_next) {
      const size_t tn = q.tok0 + static_cast<size_t>(q.nt) * p.H;
      v.dtn = to_f(dtg[tn]);
      v.lamn = to_f(lamg[tn]);
    }
  }
  return v;
}
__device__ __forceinline__ void chunk_coefs_from(const Shape& sh, const ChunkPos& q, float A, const InSmem& L,
                                                 float* sm, const CoefIn& v) {
  if (threadIdx.x < 32) {
    const int t = threadIdx.x;
    const bool ok = t < q.nt;
    const float dt = v.dt, lam = v.lam, dtn = v.dtn, lamn = v.lamn;
    float ell = dt * A;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, ell, d);
      if (t >= d) ell += u;
    }
    if (t < sh.c) {
      sm[L.dt + t] = dt;
      sm[L.lam + t] = lam;
      sm[L.ell + t] = ell;
      sm[L.el + t] = ok ? expf(ell) : 0.f;
      sm[L.gam + t] = lam * dt;
      sm[L.q + t] = (1.f - lam) * dt;
    }
    if (t == 0) sm[L.q + sh.c] = (1.f - lamn) * dtn;
  }
}
template <typename Tin>
__device__ __forceinline__ void chunk_coefs(const BwdParams& p, const Shape& sh, const ChunkPos& q, float A,
                                            const InSmem& L, float* sm) {
  chunk_coefs_from(sh, q, A, L, sm, load_coefs<Tin>(p, q));
}

// theta rows of the chunk into the th area (asynchronous copies when kV, else fp32 scalars).
template <typename Tin, bool kV>
__device__ __forceinline__ void issue_theta(const BwdParams& p, const Shape& sh, const ChunkPos& q, float* s_th) {
  const Tin* thg = static_cast<const Tin*>(p.theta);
  const int K = sh.K;
  if constexpr (kV) {
    constexpr int vec = 16 / sizeof(Tin);
    const int per = K / vec, n = q.nt * per;
    Tin* dst = reinterpret_cast<Tin*>(s_th);
    for (int e = threadIdx.x; e < n; e += blockDim.x) {
      const int t = e / per, col = (e - t * per) * vec;
      cp_async16(dst + t * K + col, thg + (q.tok0 + static_cast<size_t>(t) * p.H) * K + col);
    }
  } else {
    for (int e = threadIdx.x; e < q.nt * K; e += blockDim.x) {
      const int t = e / K;
      s_th[e] = to_f(thg[(q.tok0 + static_cast<size_t>(t) * p.H) * K + (e - t * K)]);
    }
  }
}
template <typename Tin, bool kV>
__device__ __forceinline__ float theta_at(const float* s_th, int e) {
  if constexpr (kV)
    return to_f(reinterpret_cast<const Tin*>(s_th)[e]);
  else
    return s_th[e];
}

// psi_t = sum_{u <= t} dt_u theta_u from the chunk's start, reduced to [-pi, pi] after every
// step, as cos / sin [c][K] (identity past nt); sig_out[kk] (when given) gets psi of the last
// token.  The tokens are split into G segments with one thread per (pair, segment): the
// reduced sum over each segment first, then every thread starts from the reduced sum of the
// segments before its own and steps through its tokens.  Contains a barrier: every thread of
// the CTA calls it.
template <typename Tin, bool kV>
__device__ __forceinline__ void chunk_angles(const ChunkPos& q, const Shape& sh, float* sm, const InSmem& L,
                                             const float* s_th, float* sig_out) {
  const int K = sh.K, c = sh.c, nthr = blockDim.x;
  float* s_part = sm + L.part;
  float* s_cs = sm + L.cs;
  float* s_sn = sm + L.sn;
  const int G = max(1, min(c, nthr / K)), per = (c + G - 1) / G;
  for (int e = threadIdx.x; e < K * G; e += nthr) {
    const int g = e / K, kk = e - g * K, t1 = min((g + 1) * per, q.nt);
    float ph = 0.f;
    for (int t = g * per; t < t1; ++t) ph = wrap(fmaf(sm[L.dt + t], theta_at<Tin, kV>(s_th, t * K + kk), ph));
    s_part[e] = ph;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < K * G; e += nthr) {
    const int g = e / K, kk = e - g * K, t1 = min((g + 1) * per, c);
    float ph = 0.f;
    for (int h = 0; h < g; ++h) ph = wrap(ph + s_part[h * K + kk]);
    for (int t = g * per; t < t1; ++t) {
      float sn = 0.f, cs = 1.f;
      if (t < q.nt) {
        ph = wrap(fmaf(sm[L.dt + t], theta_at<Tin, kV>(s_th, t * K + kk), ph));
        __sincosf(ph, &sn, &cs);
        if (t == q.last && sig_out) sig_out[kk] = ph;
      }
      s_cs[t * K + kk] = cs;
      s_sn[t * K + kk] = sn;
    }
  }
}

// The chunk's inputs: coefficients, theta and psi, and B~, C~ (rotated by psi), X, dY as
// fp32 rows, X rows times xscale and dY rows times yscale when given.  extra() issues further
// asynchronous copies with the inputs' (it runs after theta's copies are committed); the
// function returns with every copy landed and a barrier passed.
template <typename Tin, typename Tdy, bool kV, typename FX, typename FS>
__device__ __forceinline__ void load_chunk(const BwdParams& p, const Shape& sh, const ChunkPos& q, float A,
                                           const InSmem& L, float* sm, float* sig_out, FX extra, FS scales,
                                           bool scale_x, bool scale_y) {
  const int N = sh.N, P = sh.P, R = sh.R, c = sh.c, K = sh.K;
  const size_t ts = p.H;
  issue_theta<Tin, kV>(p, sh, q, sm + L.th);
  if constexpr (kV) cp_async_commit();
  issue_rows<Tin, kV>(static_cast<const Tin*>(p.B), q, ts, c, R, N, sm + L.Bt, L.ldN,
                      reinterpret_cast<Tin*>(sm + L.rB));
  issue_rows<Tin, kV>(static_cast<const Tin*>(p.C), q, ts, c, R, N, sm + L.Ct, L.ldN,
                      reinterpret_cast<Tin*>(sm + L.rC));
  issue_rows<Tin, kV>(static_cast<const Tin*>(p.x), q, ts, c, R, P, sm + L.X, L.ldP,
                      reinterpret_cast<Tin*>(sm + L.rX));
  issue_rows<Tdy, kV>(static_cast<const Tdy*>(p.dy), q, ts, c, R, P, sm + L.dY, L.ldP,
                      reinterpret_cast<Tdy*>(sm + L.rY));
  extra();
  if constexpr (kV) cp_async_commit();
  chunk_coefs<Tin>(p, sh, q, A, L, sm);
  if constexpr (kV) asm volatile("cp.async.wait_group 1;" ::: "memory");
  __syncthreads();
  chunk_angles<Tin, kV>(q, sh, sm, L, sm + L.th, sig_out);
  scales();  // per-row weights from the coefficients
  if constexpr (kV) cp_async_wait_all();
  __syncthreads();
  finish_rows<Tin, kV>(q, c, R, N, sm + L.Bt, L.ldN, reinterpret_cast<const Tin*>(sm + L.rB), true,
                       sm + L.cs, sm + L.sn, K, nullptr);
  finish_rows<Tin, kV>(q, c, R, N, sm + L.Ct, L.ldN, reinterpret_cast<const Tin*>(sm + L.rC), true,
                       sm + L.cs, sm + L.sn, K, nullptr);
  finish_rows<Tin, kV>(q, c, R, P, sm + L.X, L.ldP, reinterpret_cast<const Tin*>(sm + L.rX), false,
                       nullptr, nullptr, K, scale_x ? sm + L.wx : nullptr);
  finish_rows<Tdy, kV>(q, c, R, P, sm + L.dY, L.ldP, reinterpret_cast<const Tdy*>(sm + L.rY), false,
                       nullptr, nullptr, K, scale_y ? sm + L.rowel : nullptr);
  __syncthreads();
}

// Per row: wx, its weight on the exit-state terms (Mh[last, t], plus q of the next chunk's
// first token for the last token, whose trapezoid term that chunk folds in), and exp(l) of
// its token.  Needs the coefficients (a barrier after chunk_coefs).
__device__ __forceinline__ void row_weights(const ChunkPos& q, int c, int R, const InSmem& L, float* sm) {
  for (int row = threadIdx.x; row < c * R; row += blockDim.x) {
    const int t = row / R;
    float wx = 0.f;
    if (t < q.nt)
      wx = t == q.last ? sm[L.gam + t] + sm[L.q + c]
                       : expf(sm[L.ell + q.last] - sm[L.ell + t]) * (sm[L.gam + t] + sm[L.q + t + 1]);
    sm[L.wx + row] = wx;
    sm[L.rowel + row] = sm[L.el + t];
  }
}

// ------------------------------------------------------------------ chunk-local state terms
template <typename Tin, typename Tdy, bool kV, int SN, int SP, int SR, int SC>
__global__ void __launch_bounds__(kThreads, 2) bwd_local_kernel(const BwdParams p) {
  extern __shared__ __align__(16) float sm[];
  const Shape sh = shape_of<SN, SP, SR, SC>(p);
  const int N = sh.N, P = sh.P, R = sh.R, c = sh.c, M = sh.M, K = sh.K;
  const int bh = blockIdx.x / p.nch, k = blockIdx.x % p.nch;
  const ChunkPos q = chunk_pos(p, bh, k, c);
  const LocalSmem S = local_smem(N, P, R, c, sizeof(Tin), sizeof(Tdy));
  const InSmem& L = S.in;
  const size_t slot = static_cast<size_t>(bh) * p.nch + k;
  load_chunk<Tin, Tdy, kV>(p, sh, q, p.A[bh % p.H], L, sm, p.wsSig + slot * K, [] {},
                           [&] { row_weights(q, c, R, L, sm); }, true, true);
  if (threadIdx.x == 0) p.wsDec[slot] = sm[L.el + q.last];
  // dH[n][p] = sum_s B~[s][n] (wx_s X[s][p]),  dG[n][p] = sum_i C~[i][n] (exp(l_i) dY[i][p])
  float* dH = p.wsH + slot * N * P;
  float* dG = p.wsG + slot * N * P;
  int rr = 0;
  product<2, 4, 4, 4, false, false, kV>(rr, N, P, M, sm + L.Bt, L.ldN, sm + L.X, L.ldP,
                               [&](int n, int pc, float v) { dH[n * P + pc] = v; });
  product<2, 4, 4, 4, false, false, kV>(rr, N, P, M, sm + L.Ct, L.ldN, sm + L.dY, L.ldP,
                               [&](int n, int pc, float v) { dG[n * P + pc] = v; });
}

// ------------------------------------------------------------------ chunk-level scans
// One thread per (batch row, head, state pair kk, column p): rows 2 kk and 2 kk + 1 of the
// state in column p.  blockIdx.y = 0: the folded entry states Hp(k), written over dH(k);
// blockIdx.y = 1: the exit cotangents Gout(k), written over dG(k), and dh0.
template <typename Tin>
__global__ void __launch_bounds__(kThreads) bwd_scan_kernel(const BwdParams p, long long total) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const int K = p.K, P = p.P, N = p.N, NP = N * P, nch = p.nch;
  const int KP = K * P;
  const int bh = static_cast<int>(idx / KP), rem = static_cast<int>(idx - static_cast<long long>(bh) * KP);
  const int kk = rem / P, pc = rem - kk * P, n0 = 2 * kk;
  const size_t base = static_cast<size_t>(bh) * nch * NP + static_cast<size_t>(n0) * P + pc;
  const float* dec = p.wsDec + static_cast<size_t>(bh) * nch;
  const float* sig = p.wsSig + static_cast<size_t>(bh) * nch * K + kk;
  const float ph0 = p.phi0 ? wrap(p.phi0[static_cast<size_t>(bh) * K + kk]) : 0.f;
  float s0, c0;
  sincosf(ph0, &s0, &c0);
  const size_t e0 = static_cast<size_t>(bh) * NP + static_cast<size_t>(n0) * P + pc;
  if (blockIdx.y == 0) {
    // Hp(0) in chunk 0's frame: R(-phi_0) h0 + q_0 prevB^T prevx (prevB is stored unrotated,
    // which is its rotated value read in chunk 0's frame)
    float a = 0.f, b = 0.f;
    if (p.h0) {
      a = p.h0[e0];
      b = p.h0[e0 + P];
    }
    float H0 = c0 * a - s0 * b, H1 = s0 * a + c0 * b;
    if (p.prevB0 && p.prevx0) {
      const Tin* dtg = static_cast<const Tin*>(p.dt);
      const Tin* lamg = static_cast<const Tin*>(p.lam);
      const Tin* pB = static_cast<const Tin*>(p.prevB0);
      const Tin* px = static_cast<const Tin*>(p.prevx0);
      const size_t o = static_cast<size_t>(bh / p.H) * p.T * p.H + bh % p.H;
      const float q0 = (1.f - to_f(lamg[o])) * to_f(dtg[o]);
      float f0 = 0.f, f1 = 0.f;
      for (int r = 0; r < p.R; ++r) {
        const float xv = to_f(px[(static_cast<size_t>(bh) * p.R + r) * P + pc]);
        f0 = fmaf(to_f(pB[(static_cast<size_t>(bh) * p.R + r) * N + n0]), xv, f0);
        f1 = fmaf(to_f(pB[(static_cast<size_t>(bh) * p.R + r) * N + n0 + 1]), xv, f1);
      }
      H0 = fmaf(q0, f0, H0);
      H1 = fmaf(q0, f1, H1);
    }
    float* hp = p.wsH + base;
    float d0 = hp[0], d1 = hp[P];
    for (int k = 0; k < nch; ++k) {
      float n0v = 0.f, n1v = 0.f;
      if (k + 1 < nch) {
        n0v = hp[static_cast<size_t>(k + 1) * NP];
        n1v = hp[static_cast<size_t>(k + 1) * NP + P];
      }
      hp[static_cast<size_t>(k) * NP] = H0;
      hp[static_cast<size_t>(k) * NP + P] = H1;
      if (k + 1 < nch) {
        const float dk = dec[k];
        float sn, cs;
        sincosf(sig[static_cast<size_t>(k) * K], &sn, &cs);
        const float X0 = fmaf(dk, H0, d0), X1 = fmaf(dk, H1, d1);
        H0 = cs * X0 - sn * X1;
        H1 = sn * X0 + cs * X1;
      }
      d0 = n0v;
      d1 = n1v;
    }
  } else {
    // the angle before the last chunk turns the exit cotangent into that chunk's frame
    float ph = ph0;
    for (int k = 0; k + 1 < nch; ++k) ph = wrap(ph + sig[static_cast<size_t>(k) * K]);
    float sn, cs;
    sincosf(ph, &sn, &cs);
    float a = 0.f, b = 0.f;
    if (p.dhT) {
      a = p.dhT[e0];
      b = p.dhT[e0 + P];
    }
    float G0 = cs * a - sn * b, G1 = sn * a + cs * b;
    float* gp = p.wsG + base;
    float d0 = gp[static_cast<size_t>(nch - 1) * NP], d1 = gp[static_cast<size_t>(nch - 1) * NP + P];
    for (int k = nch - 1; k >= 0; --k) {
      float n0v = 0.f, n1v = 0.f;
      if (k > 0) {
        n0v = gp[static_cast<size_t>(k - 1) * NP];
        n1v = gp[static_cast<size_t>(k - 1) * NP + P];
      }
      gp[static_cast<size_t>(k) * NP] = G0;
      gp[static_cast<size_t>(k) * NP + P] = G1;
      const float dk = dec[k];
      const float Y0 = fmaf(dk, G0, d0), Y1 = fmaf(dk, G1, d1);  // dHp(k), chunk k's frame
      if (k > 0) {
        sincosf(sig[static_cast<size_t>(k - 1) * K], &sn, &cs);
        G0 = cs * Y0 + sn * Y1;
        G1 = cs * Y1 - sn * Y0;
      } else {
        p.wsDH0[e0] = Y0;
        p.wsDH0[e0 + P] = Y1;
        if (p.dh0) {  // back to the absolute frame: R(phi_0)
          p.dh0[e0] = c0 * Y0 + s0 * Y1;
          p.dh0[e0 + P] = c0 * Y1 - s0 * Y0;
        }
      }
      d0 = n0v;
      d1 = n1v;
    }
  }
}

// ------------------------------------------------------------------ per-chunk adjoint
// kTS: Hp and Gout arrive by TMA tensor copies (p.tmH, p.tmG) in the swizzled layout of swz(),
// completing on an mbarrier, instead of 16-byte thread copies into padded rows (P % 32 == 0).
template <typename Tin, typename Tdy, bool kV, int SN, int SP, int SR, int SC, int NT, bool kTS>
__global__ void __launch_bounds__(NT, 1) bwd_chunk_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ __align__(16) float sm_raw[];
  // the base at a 1024-byte boundary (the swizzled copies' destinations need it)
  float* sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u) / 4u;
  const Shape sh = shape_of<SN, SP, SR, SC>(p);
  const int N = sh.N, P = sh.P, R = sh.R, c = sh.c, M = sh.M, K = sh.K, NP = N * P;
  const int ldN = N + kPad, ldP = P + kPad, ldM = M + kPad, ldT = c + 1;  // = L.ldN, L.ldP
  const ChunkSmem S = chunk_smem(N, P, R, c, sizeof(Tin), sizeof(Tdy), kTS);
  const InSmem& L = S.in;
  const size_t tstride = p.H;
  const int total = p.BH * p.nch;
  float* sBt = sm + L.Bt;
  float* sCt = sm + L.Ct;
  float* sX = sm + L.X;
  float* sdY = sm + L.dY;
  float* sQ = sm + S.Q;
  float* sXG = sm + S.XG;
  float* sW = sm + S.W;
  float* sHp = sm + S.Hp;
  float* sGo = sm + S.Go;
  float* sS = sm + S.S;
  float* sE = sm + S.E;
  float* sdphi = sm + S.dphi;
  float* s_Mh = sm + S.Mh;
  float* s_ex = sm + S.ex;
  float* s_dM = sm + S.dM;
  float* s_dexp = sm + S.dexp;
  float* s_wdot = sm + S.wdot;
  float* s_dell = sm + S.dell;
  float* s_dgam = sm + S.dgam;
  float* s_dq = sm + S.dq;
  float* s_red = sm + S.red;
  const float* s_dt = sm + L.dt;
  const float* s_lam = sm + L.lam;
  const float* s_ell = sm + L.ell;
  const float* s_el = sm + L.el;
  const float* s_gam = sm + L.gam;
  const float* s_q = sm + L.q;
  const float* s_wx = sm + L.wx;
  const float* s_rowel = sm + L.rowel;
  const float* s_cs = sm + L.cs;
  const float* s_sn = sm + L.sn;
  float* s_th = sm + S.th;
  const Tin* thg = static_cast<const Tin*>(p.theta);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  // a chunk's Hp and Gout into their areas (asynchronous copies when kV)
  const uint32_t s_bar = smem_u32(sm + S.bar);
  auto fetch_state = [&](size_t slot_) {
    const float* hp = p.wsH + slot_ * NP;
    const float* go = p.wsG + slot_ * NP;
    if constexpr (kTS) {
      if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(s_bar, 2u * static_cast<uint32_t>(NP) * 4u);
        for (int bx = 0; bx < P / 32; ++bx) {
          tma_load_2d(smem_u32(sHp + bx * N * 32), &p.tmH, s_bar, 32 * bx, static_cast<int>(slot_) * N);
          tma_load_2d(smem_u32(sGo + bx * N * 32), &p.tmG, s_bar, 32 * bx, static_cast<int>(slot_) * N);
        }
      }
    } else if constexpr (kV) {
      const int per = P / 4;
      for (int e = threadIdx.x; e < N * per; e += blockDim.x) {
        const int n = e / per, col = (e - n * per) * 4;
        cp_async16(sHp + n * ldP + col, hp + n * P + col);
        cp_async16(sGo + n * ldP + col, go + n * P + col);
      }
    } else {
      for (int e = threadIdx.x; e < NP; e += blockDim.x) {
        const int n = e / P, col = e - n * P;
        sHp[n * ldP + col] = hp[e];
        sGo[n * ldP + col] = go[e];
      }
    }
  };
  auto pos_of = [&](int j) { return chunk_pos(p, j / p.nch, j % p.nch, c); };

  // Persistent: CTA b takes chunks b, b + gridDim.x, ...; theta, Hp, Gout, dt and lambda of the
  // next chunk are requested while the current one finishes (their areas are free by then).
  CoefIn cin{0.f, 0.f, 0.f, 0.f, 0.f};
  if constexpr (kTS) {
    if (threadIdx.x == 0) {
      mbar_init(s_bar, 1);
      fence_mbar_init();
    }
    __syncthreads();
  }
  if (static_cast<int>(blockIdx.x) < total) {
    const ChunkPos q0 = pos_of(blockIdx.x);
    issue_theta<Tin, kV>(p, sh, q0, s_th);
    fetch_state(blockIdx.x);
    if constexpr (kV) cp_async_commit();
    cin = load_coefs<Tin>(p, q0);
  }
  for (int j = blockIdx.x, it = 0; j < total; j += gridDim.x, ++it) {
  const ChunkPos q = pos_of(j);
  const size_t slot = j;
  const float A = cin.A;  // (warp 0 only: the coefficients and d dt use it)

  // ---------------------------------------------------------------- inputs of the chunk
  issue_rows<Tin, kV>(static_cast<const Tin*>(p.B), q, tstride, c, R, N, sBt, ldN, reinterpret_cast<Tin*>(sm + L.rB));
  issue_rows<Tin, kV>(static_cast<const Tin*>(p.C), q, tstride, c, R, N, sCt, ldN, reinterpret_cast<Tin*>(sm + L.rC));
  issue_rows<Tin, kV>(static_cast<const Tin*>(p.x), q, tstride, c, R, P, sX, ldP, reinterpret_cast<Tin*>(sm + L.rX));
  issue_rows<Tdy, kV>(static_cast<const Tdy*>(p.dy), q, tstride, c, R, P, sdY, ldP, reinterpret_cast<Tdy*>(sm + L.rY));
  if constexpr (kV) cp_async_commit();
  chunk_coefs_from(sh, q, A, L, sm, cin);
  if constexpr (kV) asm volatile("cp.async.wait_group 1;" ::: "memory");  // theta (and Hp, Gout)
  if constexpr (kTS) {
    // Hp and Gout: a wait that runs out (bounded) ends the CTA's work and is reported
    if (!__syncthreads_and(mbar_wait(s_bar, static_cast<uint32_t>(it) & 1u))) {
      if (threadIdx.x == 0) atomicOr(p.status, kDevTimeout);
      break;
    }
  } else {
    __syncthreads();
  }
  chunk_angles<Tin, kV>(q, sh, sm, L, s_th, nullptr);
  row_weights(q, c, R, L, sm);
  if constexpr (kV) cp_async_wait_all();
  __syncthreads();
  finish_rows<Tin, kV>(q, c, R, N, sBt, ldN, reinterpret_cast<const Tin*>(sm + L.rB), true, s_cs, s_sn, K, nullptr);
  finish_rows<Tin, kV>(q, c, R, N, sCt, ldN, reinterpret_cast<const Tin*>(sm + L.rC), true, s_cs, s_sn, K, nullptr);
  finish_rows<Tin, kV>(q, c, R, P, sX, ldP, reinterpret_cast<const Tin*>(sm + L.rX), false, nullptr, nullptr, K, nullptr);
  finish_rows<Tdy, kV>(q, c, R, P, sdY, ldP, reinterpret_cast<const Tdy*>(sm + L.rY), false, nullptr, nullptr, K, nullptr);
  __syncthreads();

  // ---------------------------------------------------------------- products with the inputs
  // tables per token pair: exp(l_i - l_s) and Mh[i, s]
  for (int e = threadIdx.x; e < c * c; e += blockDim.x) {
    const int ti = e / c, ts = e - ti * c;
    float ex = 0.f, m = 0.f;
    if (ts <= ti && ti < q.nt) {
      ex = expf(s_ell[ti] - s_ell[ts]);
      m = ts == ti ? s_gam[ti] : ex * (s_gam[ts] + s_q[ts + 1]);
    }
    s_ex[ti * ldT + ts] = ex;
    s_Mh[ti * ldT + ts] = m;
  }
  {  // <Gout, Hp>, one partial per thread (both states in the same layout)
    float gh = 0.f;
    for (int e = threadIdx.x; e < NP; e += blockDim.x) {
      const int n = e / P, col = e - n * P;
      const int o = kTS ? e : n * ldP + col;
      gh = fmaf(sGo[o], sHp[o], gh);
    }
    s_red[threadIdx.x] = gh;
  }
  int rr = 0;
  // W = B~ Gout, S = C~ B~^T, Q = dY Hp^T, XG = X Gout^T, E = dY X^T (tiles of about equal
  // work, the largest products first)
  auto state_product = [&](auto kbk, int NJd, int NK, const float* a, int lda, const float* st, auto out) {
    constexpr bool kBK = decltype(kbk)::value;
    if constexpr (kTS)
      gemm_tc<2, kBK ? 2 : 2, true, kBK, true>(rr, M, NJd, NK, a, lda, st, N, out);
    else
      product<2, 2, kBK ? 4 : 2, 4, true, kBK, kV>(rr, M, NJd, NK, a, lda, st, ldP, out);
  };
  state_product(std::false_type{}, P, N, sBt, ldN, sGo,
                [&](int s_, int pc, float v) { sW[s_ * ldP + pc] = v; });
  product<2, 2, 2, 4, true, true, kV>(rr, M, M, N, sCt, ldN, sBt, ldN,
                             [&](int i, int s_, float v) { sS[i * ldM + s_] = v; });
  state_product(std::true_type{}, N, P, sdY, ldP, sHp, [&](int i, int n, float v) { sQ[i * ldN + n] = v; });
  state_product(std::true_type{}, N, P, sX, ldP, sGo, [&](int s_, int n, float v) { sXG[s_ * ldN + n] = v; });
  product<2, 2, 2, 4, true, true, kV>(rr, M, M, P, sdY, ldP, sX, ldP,
                             [&](int i, int s_, float v) { sE[i * ldM + s_] = v; });
  if constexpr (kTS) fence_proxy_async_smem();  // the reads of Hp and Gout before the TMA rewrites them
  __syncthreads();
  // Hp and Gout are read: the next chunk's may come in
  const int jn = j + static_cast<int>(gridDim.x);
  ChunkPos qn{};
  if (jn < total) {
    qn = pos_of(jn);
    fetch_state(jn);
    cin = load_coefs<Tin>(p, qn);
  }

  // ---------------------------------------------------------------- per token and token pair
  // per token (a warp each): wdot_t = sum over its rows of <W, X> (= <Gout, B~_t^T X_t>),
  // dexp_t = sum over its rows of <C~, Q> (+ <Gout, Hp> at the last token)
  for (int t = warp; t < c; t += nw) {
    float a = 0.f, b = 0.f;
    if (t < q.nt) {
      for (int e = lane; e < R * P; e += 32) {
        const int row = t * R + e / P, col = e % P;
        a = fmaf(sW[row * ldP + col], sX[row * ldP + col], a);
      }
      for (int e = lane; e < R * N; e += 32) {
        const int row = t * R + e / N, col = e % N;
        b = fmaf(sCt[row * ldN + col], sQ[row * ldN + col], b);
      }
      if (t == q.last)
        for (int i = lane; i < static_cast<int>(blockDim.x); i += 32) b += s_red[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a += __shfl_xor_sync(0xffffffffu, a, o);
      b += __shfl_xor_sync(0xffffffffu, b, o);
    }
    if (lane == 0) {
      s_wdot[t] = a;
      s_dexp[t] = b;
    }
  }
  // dMh per token pair (its R x R entries of S o E), then Mh o S and Mh o E in place
  for (int e = threadIdx.x; e < c * c; e += blockDim.x) {
    const int ti = e / c, ts = e - ti * c;
    const float m = s_Mh[ti * ldT + ts];
    float v = 0.f;
    for (int r = 0; r < R; ++r)
      for (int r2 = 0; r2 < R; ++r2) {
        const int o = (ti * R + r) * ldM + ts * R + r2;
        const float sv = sS[o], ev = sE[o];
        v = fmaf(sv, ev, v);
        sS[o] = m * sv;
        sE[o] = m * ev;
      }
    s_dM[ti * ldT + ts] = ts <= ti && ti < q.nt ? v : 0.f;
  }
  __syncthreads();

  // ---------------------------------------------------------------- gradients of the rows
  rr = 0;
  // dC~ = (Mh o E) B~ + exp(l) Q, over Q
  product<2, 2, 2, 4, true, false, kV>(rr, M, N, M, sE, ldM, sBt, ldN, [&](int i, int n, float v) {
    sQ[i * ldN + n] = fmaf(s_rowel[i], sQ[i * ldN + n], v);
  });
  // dB~ = (Mh o E)^T C~ + wx X Gout^T, over XG
  product<2, 2, 2, 4, false, false, kV>(rr, M, N, M, sE, ldM, sCt, ldN, [&](int s_, int n, float v) {
    sXG[s_ * ldN + n] = fmaf(s_wx[s_], sXG[s_ * ldN + n], v);
  });
  // dX = (Mh o S)^T dY + wx W, to global
  float* dxg = p.dx;
  product<2, 2, 2, 4, false, false, kV>(rr, M, P, M, sS, ldM, sdY, ldP, [&](int s_, int pc, float v) {
    const int ts = s_ / R;
    if (ts < q.nt)
      dxg[(q.tok0 + static_cast<size_t>(ts) * tstride) * R * P + static_cast<size_t>(s_ - ts * R) * P + pc] =
          fmaf(s_wx[s_], sW[s_ * ldP + pc], v);
  });
  __syncthreads();
  // S and E are read: the next chunk's theta may come in
  if (jn < total) issue_theta<Tin, kV>(p, sh, qn, s_th);
  if constexpr (kV) cp_async_commit();

  // ---------------------------------------------------------------- rotation adjoint
  // the mask and fold parameters per token, a warp each, lanes over the other token (the last
  // row of dMh also carries the exit term <Gout, B~_s^T X_s> = wdot_s)
  for (int t = warp; t < c; t += nw) {
    auto dMf = [&](int ti, int ts) { return s_dM[ti * ldT + ts] + (ti == q.last ? s_wdot[ts] : 0.f); };
    const int j = lane;
    float rw = 0.f, cl = 0.f, cg = 0.f, cq = 0.f;
    if (t < q.nt && j < q.nt) {
      if (j < t) rw = dMf(t, j) * s_Mh[t * ldT + j];  // row t: l_t
      if (j > t) {                                    // column t: l_t, gamma_t (through w_t)
        const float d = dMf(j, t);
        cl = d * s_Mh[j * ldT + t];
        cg = d * s_ex[j * ldT + t];
      }
      if (t > 0 && j >= t) cq = dMf(j, t - 1) * s_ex[j * ldT + t - 1];  // q_t weighs column t - 1
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      rw += __shfl_xor_sync(0xffffffffu, rw, o);
      cl += __shfl_xor_sync(0xffffffffu, cl, o);
      cg += __shfl_xor_sync(0xffffffffu, cg, o);
      cq += __shfl_xor_sync(0xffffffffu, cq, o);
    }
    if (lane == 0) {
      const bool ok = t < q.nt;
      s_dell[t] = ok ? fmaf(s_dexp[t], s_el[t], rw - cl) : 0.f;
      s_dgam[t] = ok ? cg + dMf(t, t) : 0.f;
      s_dq[t] = ok ? cq : 0.f;  // q_0's fold term is added later
    }
  }
  // the rotation adjoint
  float* dBg = p.dB;
  float* dCg = p.dC;
  for (int e = threadIdx.x; e < q.nt * K; e += blockDim.x) {  // a (token, pair), its R rows in order
    const int t = e / K, kk = e - t * K;
    const float cs = s_cs[t * K + kk], sn = s_sn[t * K + kk];
    float dph = 0.f;
    for (int r = 0; r < R; ++r) {
      const int row = t * R + r;
      const float db0 = sXG[row * ldN + 2 * kk], db1 = sXG[row * ldN + 2 * kk + 1];
      const float dc0 = sQ[row * ldN + 2 * kk], dc1 = sQ[row * ldN + 2 * kk + 1];
      const float b0 = sBt[row * ldN + 2 * kk], b1 = sBt[row * ldN + 2 * kk + 1];
      const float c0 = sCt[row * ldN + 2 * kk], c1 = sCt[row * ldN + 2 * kk + 1];
      const size_t o = ((q.tok0 + static_cast<size_t>(t) * tstride) * R + r) * N + 2 * kk;
      *reinterpret_cast<float2*>(dBg + o) = make_float2(cs * db0 - sn * db1, sn * db0 + cs * db1);
      *reinterpret_cast<float2*>(dCg + o) = make_float2(cs * dc0 - sn * dc1, sn * dc0 + cs * dc1);
      dph += db0 * b1 - db1 * b0 + dc0 * c1 - dc1 * c0;
    }
    sdphi[t * K + kk] = dph;
  }
  if (threadIdx.x == 0 && q.has_next) p.wsDqf[slot + 1] = s_wdot[q.last];  // next chunk's fold
  __syncthreads();
  // chunk-local suffix sums of d phi: this chunk's part of d theta, and the chunk's total.  The
  // tokens are split into G segments, one thread per (pair, segment): each segment's sum, then
  // every thread starts from the sum of the later segments and walks its tokens backwards.
  {
    const int G = max(1, min(c, static_cast<int>(blockDim.x) / K)), per = (c + G - 1) / G;
    for (int e = threadIdx.x; e < K * G; e += blockDim.x) {
      const int g = e / K, kk = e - g * K, t1 = min((g + 1) * per, q.nt);
      float v = 0.f;
      for (int t = g * per; t < t1; ++t) v += sdphi[t * K + kk];
      s_red[e] = v;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < K * G; e += blockDim.x) {
      const int g = e / K, kk = e - g * K, t1 = min((g + 1) * per, q.nt), tb = g * per;
      float v = 0.f;
      for (int h = G - 1; h > g; --h) v += s_red[h * K + kk];
      for (int ta = t1 - 1; ta >= tb; ta -= 4) {  // theta (from global) four tokens at a time
        float th[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          th[u] = ta - u >= tb ? to_f(thg[(q.tok0 + static_cast<size_t>(ta - u) * tstride) * K + kk]) : 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int t = ta - u;
          if (t >= tb) {
            v += sdphi[t * K + kk];
            p.dtheta[(q.tok0 + static_cast<size_t>(t) * tstride) * K + kk] = s_dt[t] * v;
            sdphi[t * K + kk] = v * th[u];  // theta . suffix, summed below
          }
        }
      }
      if (g == 0) p.wsSphi[slot * K + kk] = v;
    }
  }
  __syncthreads();
  // per token: the angle term of d dt (a warp per token, pairs in a fixed order)
  for (int t = warp; t < q.nt; t += nw) {
    float v = 0.f;
    for (int kk = lane; kk < K; kk += 32) v += sdphi[t * K + kk];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) s_dexp[t] = v;  // (dexp is no longer read)
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int t = threadIdx.x;
    // d a_t = sum_{i >= t} d l_i (l_i = sum_{s <= i} a_s within the chunk)
    float da = t < q.nt ? s_dell[t] : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float v = __shfl_down_sync(0xffffffffu, da, o);
      if (t + o < 32) da += v;
    }
    float dadt = 0.f;
    if (t < q.nt) {
      const float dt = s_dt[t], lam = s_lam[t];
      const size_t o = q.tok0 + static_cast<size_t>(t) * tstride;
      p.ddt[o] = s_dexp[t] + da * A + lam * s_dgam[t] + (1.f - lam) * s_dq[t];
      p.dlam[o] = dt * (s_dgam[t] - s_dq[t]);
      dadt = da * dt;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dadt += __shfl_xor_sync(0xffffffffu, dadt, o);
    if (t == 0) p.wsDa[slot] = dadt;
  }
  __syncthreads();  // the next chunk's inputs overwrite this one's
  }
  if constexpr (kV) cp_async_wait_all();
}

// ------------------------------------------------------------------ carries across chunks
// One CTA per (batch row, head): the d phi sums over chunks turned into sums over the chunks
// after each one (in place), the (b, h) part of dA, and the fold gradient of the sequence's
// first token, <dHp(0), prevB^T prevx> (chunk 0's frame, where prevB reads unrotated).
template <typename Tin>
__global__ void __launch_bounds__(kThreads) bwd_carry_kernel(const BwdParams p) {
  __shared__ float scratch[kThreads];
  const int bh = blockIdx.x, K = p.K, nch = p.nch, N = p.N, P = p.P, R = p.R;
  for (int kk = threadIdx.x; kk < K; kk += blockDim.x) {
    float carry = 0.f;
    for (int k = nch - 1; k >= 0; --k) {
      float* s = p.wsSphi + (static_cast<size_t>(bh) * nch + k) * K + kk;
      const float v = *s;
      *s = carry;
      carry += v;
    }
  }
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int k = 0; k < nch; ++k) s += p.wsDa[static_cast<size_t>(bh) * nch + k];
    p.dApart[bh] = s;
  }
  float f = 0.f;
  if (p.prevB0 && p.prevx0) {
    const Tin* pB = static_cast<const Tin*>(p.prevB0) + static_cast<size_t>(bh) * R * N;
    const Tin* px = static_cast<const Tin*>(p.prevx0) + static_cast<size_t>(bh) * R * P;
    const float* g = p.wsDH0 + static_cast<size_t>(bh) * N * P;
    for (int e = threadIdx.x; e < N * P; e += blockDim.x) {
      const int n = e / P, pc = e - n * P;
      float w = 0.f;
      for (int r = 0; r < R; ++r) w = fmaf(to_f(pB[r * N + n]), to_f(px[r * P + pc]), w);
      f = fmaf(g[e], w, f);
    }
  }
  f = block_sum(f, scratch);
  if (threadIdx.x == 0) p.wsDqf[static_cast<size_t>(bh) * nch] = f;
}

// One CTA per (batch row, head, chunk): d theta_t += dt_t carry, d dt_t += <theta_t, carry>
// with carry the d phi of the chunks after this one; the chunk's first token takes its fold
// gradient: d dt += (1 - lambda) dq, d lambda -= dt dq.  kQ: K / 4 divides 32 and the pairs are
// taken four at a time (16-byte loads and stores), the K / 4 lanes of a token in one warp.
template <typename Tin, bool kQ>
__global__ void __launch_bounds__(kThreads) bwd_apply_kernel(const BwdParams p) {
  const int bh = blockIdx.x / p.nch, k = blockIdx.x % p.nch;
  const ChunkPos q = chunk_pos(p, bh, k, p.c);
  const int K = p.K;
  const size_t slot = static_cast<size_t>(bh) * p.nch + k;
  const Tin* dtg = static_cast<const Tin*>(p.dt);
  const Tin* lamg = static_cast<const Tin*>(p.lam);
  const Tin* thg = static_cast<const Tin*>(p.theta);
  const float* carry = p.wsSphi + slot * K;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  // the token's fold gradient and angle term, added by the lane that owns its first pairs
  auto finish = [&](int t, float v) {
    const size_t o = q.tok0 + static_cast<size_t>(t) * p.H;
    float g = p.ddt[o] + v;
    if (t == 0) {
      const float dq = p.wsDqf[slot], dt = to_f(dtg[o]), lam = to_f(lamg[o]);
      g = fmaf(1.f - lam, dq, g);
      p.dlam[o] = fmaf(-dt, dq, p.dlam[o]);
    }
    p.ddt[o] = g;
  };
  if constexpr (kQ) {
    const int KQ = K / 4, n = q.nt * KQ;
    for (int e0 = 0; e0 < n; e0 += blockDim.x) {
      const int e = e0 + threadIdx.x, t = e / KQ, j = e - t * KQ;
      float v = 0.f;
      if (e < n && q.has_next) {
        const size_t o = q.tok0 + static_cast<size_t>(t) * p.H;
        const float4 cr = *reinterpret_cast<const float4*>(carry + 4 * j);
        float th[4];
        if constexpr (sizeof(Tin) == 4) {
          const float4 tv = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(thg) + o * K + 4 * j);
          th[0] = tv.x, th[1] = tv.y, th[2] = tv.z, th[3] = tv.w;
        } else {
          const uint2 tv = *reinterpret_cast<const uint2*>(thg + o * K + 4 * j);
          const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&tv.x));
          const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&tv.y));
          th[0] = lo.x, th[1] = lo.y, th[2] = hi.x, th[3] = hi.y;
        }
        const float dt = to_f(dtg[o]);
        float4* dth = reinterpret_cast<float4*>(p.dtheta + o * K + 4 * j);
        float4 d = *dth;
        d.x = fmaf(dt, cr.x, d.x);
        d.y = fmaf(dt, cr.y, d.y);
        d.z = fmaf(dt, cr.z, d.z);
        d.w = fmaf(dt, cr.w, d.w);
        *dth = d;
        v = fmaf(th[0], cr.x, fmaf(th[1], cr.y, fmaf(th[2], cr.z, th[3] * cr.w)));
      }
      for (int o = KQ / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (e < n && j == 0) finish(t, v);
    }
  } else {
    if (q.has_next) {
      for (int e = threadIdx.x; e < q.nt * K; e += blockDim.x) {
        const int t = e / K, kk = e - t * K;
        const size_t o = q.tok0 + static_cast<size_t>(t) * p.H;
        p.dtheta[o * K + kk] = fmaf(to_f(dtg[o]), carry[kk], p.dtheta[o * K + kk]);
      }
    }
    for (int t = warp; t < q.nt; t += nw) {
      const size_t o = q.tok0 + static_cast<size_t>(t) * p.H;
      float v = 0.f;
      if (q.has_next)
        for (int kk = lane; kk < K; kk += 32) v = fmaf(to_f(thg[o * K + kk]), carry[kk], v);
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
      if (lane == 0) finish(t, v);
    }
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

int dtype_bytes(int dt) { return dt == M3_BF16 ? 2 : 4; }

// Tokens per chunk: the largest of 32, 16, 8, 4, 2, 1 with at most 64 (token, rank) rows whose
// shared memory fits one CTA of either per-chunk kernel.
constexpr size_t kSmemLimit = 227 * 1024;
int plan_c(const m3_dims& d) {
  if (d.N * d.P > 8192 || d.N % 2 || d.N > 2 * kThreadsChunk) return 0;
  const int si = dtype_bytes(d.in_dtype), sy = dtype_bytes(d.out_dtype);
  for (int c = kMaxTok; c >= 1; c /= 2) {
    if (c * d.R > kMaxRows) continue;
    if (static_cast<size_t>(chunk_smem(d.N, d.P, d.R, c, si, sy).total) * 4 + 1024 <= kSmemLimit &&
        static_cast<size_t>(local_smem(d.N, d.P, d.R, c, si, sy).total) * 4 <= kSmemLimit)
      return c;
  }
  return 0;
}

bool aligned16(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// A chunk-state array [rows][P] fp32 as a 2-D tensor map with boxes of {32 columns, N rows} and
// the 128-byte swizzle (32 fp32 columns are exactly 128 bytes).
bool state_map(CUtensorMap* m, float* base, size_t rows, int P, int N) {
  auto fn = tmap_encoder();
  if (!fn || P % 32 != 0 || N > 256) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(P), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(P) * 4};
  const cuuint32_t box[2] = {32u, static_cast<cuuint32_t>(N)};
  const cuuint32_t es[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename Tin, typename Tdy, bool kV, int SN, int SP, int SR, int SC, bool kTS = false>
cudaError_t launch_chunk_kernels(const BwdParams& p, size_t bhn, cudaStream_t s) {
  const size_t sm1 = static_cast<size_t>(local_smem(p.N, p.P, p.R, p.c, sizeof(Tin), sizeof(Tdy)).total) * 4;
  // (+ 1024: the adjoint kernel aligns its base to 1024 bytes)
  const size_t sm3 =
      static_cast<size_t>(chunk_smem(p.N, p.P, p.R, p.c, sizeof(Tin), sizeof(Tdy), kTS).total) * 4 + 1024;
  auto k1 = bwd_local_kernel<Tin, Tdy, kV, SN, SP, SR, SC>;
  // 512 threads for the shapes specialised at compile time; 256 for the others, whose runtime
  // dimensions need more registers than 512 threads leave (128 each)
  constexpr int NT = SN ? kThreadsChunk : kThreads;
  auto k3 = bwd_chunk_kernel<Tin, Tdy, kV, SN, SP, SR, SC, NT, kTS>;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k3, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3)) != cudaSuccess)
    return e;
  const unsigned nblk = static_cast<unsigned>(bhn * p.nch);
  k1<<<nblk, kThreads, sm1, s>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const long long total = static_cast<long long>(bhn) * p.K * p.P;
  bwd_scan_kernel<Tin><<<dim3(static_cast<unsigned>((total + kThreads - 1) / kThreads), 2), kThreads, 0, s>>>(p, total);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // the adjoint kernel is persistent: one CTA per SM (its shared memory admits one)
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const unsigned grid3 = nblk < static_cast<unsigned>(sms) ? nblk : static_cast<unsigned>(sms);
  k3<<<grid3, NT, sm3, s>>>(p);
  return cudaGetLastError();
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
  p.wsH = reinterpret_cast<float*>(a.ws + w.off_h);
  p.wsG = reinterpret_cast<float*>(a.ws + w.off_g);
  p.wsSig = reinterpret_cast<float*>(a.ws + w.off_sig);
  p.wsDec = reinterpret_cast<float*>(a.ws + w.off_dec);
  p.wsDH0 = reinterpret_cast<float*>(a.ws + w.off_dh0);
  p.wsSphi = reinterpret_cast<float*>(a.ws + w.off_sphi);
  p.wsDa = reinterpret_cast<float*>(a.ws + w.off_da_chunk);
  p.wsDqf = reinterpret_cast<float*>(a.ws + w.off_dqf);
  p.dApart = reinterpret_cast<float*>(a.ws + w.off_da);
  p.status = reinterpret_cast<unsigned*>(a.ws);  // the status word at the workspace start
  p.T = d.T;
  p.H = d.H;
  p.N = d.N;
  p.P = d.P;
  p.R = d.R;
  p.c = w.c;
  p.M = w.c * d.R;
  p.nch = w.nch;
  p.K = d.N / 2;
  p.BH = static_cast<int>(bhn);
  // the call's device status starts clear (m3_ssm_device_status reads it)
  if ((e = cudaMemsetAsync(a.ws, 0, sizeof(unsigned), s)) != cudaSuccess) return e;
  // 16-byte copies and tensor-core products: row lengths of 16 bytes' multiples, aligned operands,
  // (token, rank) rows a multiple of 16
  const bool vec = d.N % 16 == 0 && d.P % 8 == 0 && p.M % 16 == 0 && aligned16(a.x) && aligned16(a.B) &&
                   aligned16(a.C) && aligned16(a.theta) && aligned16(a.dy);
  // shapes with kernels specialised at compile time: SISO N 128 P 64 and MIMO rank 4 N 64 P 64
  // for them, the chunk states go by TMA tensor copies when the maps can be made
  const size_t srows = bhn * static_cast<size_t>(w.nch) * d.N;
  const bool tmaps = vec && srows < (size_t(1) << 31) && state_map(&p.tmH, p.wsH, srows, d.P, d.N) &&
                     state_map(&p.tmG, p.wsG, srows, d.P, d.N);
  if (tmaps && d.N == 128 && d.P == 64 && d.R == 1 && w.c == 32)
    e = launch_chunk_kernels<Tin, Tdy, true, 128, 64, 1, 32, true>(p, bhn, s);
  else if (tmaps && d.N == 64 && d.P == 64 && d.R == 4 && w.c == 16)
    e = launch_chunk_kernels<Tin, Tdy, true, 64, 64, 4, 16, true>(p, bhn, s);
  else if (vec && d.N == 128 && d.P == 64 && d.R == 1 && w.c == 32)
    e = launch_chunk_kernels<Tin, Tdy, true, 128, 64, 1, 32>(p, bhn, s);
  else if (vec && d.N == 64 && d.P == 64 && d.R == 4 && w.c == 16)
    e = launch_chunk_kernels<Tin, Tdy, true, 64, 64, 4, 16>(p, bhn, s);
  else if (vec)
    e = launch_chunk_kernels<Tin, Tdy, true, 0, 0, 0, 0>(p, bhn, s);
  else
    e = launch_chunk_kernels<Tin, Tdy, false, 0, 0, 0, 0>(p, bhn, s);
  if (e != cudaSuccess) return e;
  bwd_carry_kernel<Tin><<<static_cast<unsigned>(bhn), kThreads, 0, s>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int KQ = p.K / 4;
  if (p.K % 4 == 0 && KQ <= 32 && (32 % KQ) == 0)
    bwd_apply_kernel<Tin, true><<<static_cast<unsigned>(bhn * w.nch), kThreads, 0, s>>>(p);
  else
    bwd_apply_kernel<Tin, false><<<static_cast<unsigned>(bhn * w.nch), kThreads, 0, s>>>(p);
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
  w.off_dec = w.off_da_chunk + up(bh * nch * sizeof(float));
  w.off_dqf = w.off_dec + up(bh * nch * sizeof(float));
  w.off_sig = w.off_dqf + up(bh * nch * sizeof(float));
  w.off_sphi = w.off_sig + up(bh * nch * K * sizeof(float));
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
