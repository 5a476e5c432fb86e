// Chunked prefill of the Mamba-3 SSM core on sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// The method (paper section 2.3, Eq. (7) and Remark 5; section 3.3, "chunked
// MIMO: parallel within a chunk, recurrent across chunks"): inside a chunk the
// output is a masked matrix product whose mask is the 1-semiseparable decay
// mask times the 2-band convolution matrix of the trapezoid.  Writing
// l_i = sum_{k<=i} dt_k A (chunk-local), gamma_i = lambda_i dt_i and
// q_i = (1 - lambda_i) dt_i, that product is
//     M[i, j] = exp(l_i - l_j) w_j  (j < i),   M[i, i] = gamma_i,   0 (j > i),
//     w_j = gamma_j + q_{j+1},
// because beta_{j+1} = q_{j+1} alpha_{j+1} and alpha_{j+1} = exp(l_{j+1} - l_j).
// With H the state carried into the chunk (the previous chunk's last-token
// term already folded in), per chunk of 128 (token, rank) rows:
//     S = C~ B~^T                                   (GEMM1, 128 x 128 x N)
//     Y = (M (x) J_R o S) X + diag(e^{l}) C~ H      (GEMM2, GEMM3)
//     H <- e^{l_last} H + B~^T diag(d) X,  d_j = e^{l_last - l_j} w_j   (GEMM4)
// where w of the chunk's last token takes q of the next chunk's first token,
// which carries the trapezoid's previous-token term across the boundary.
// B~, C~ are B, C rotated by the cumulative angle (Proposition 3).
//
// Kernel design: one CTA per (batch row, head) sequence, 10 warps with fixed roles,
// chunks flow through a two-stage pipeline so that loads, CUDA-core work and
// tensor-core work of neighbouring chunks overlap:
//   warp 0      TMA producer: raw bf16 tiles of B, C and X (128-byte swizzle) into
//               one of two stages.
//   warp 1      MMA issuer (one thread): GEMM1, GEMM4, GEMM3, GEMM2 per chunk.
//   warps 2-5   transform: discretisation (decay log-sums, trapezoid weights), the
//               cumulative angle, rotation of B and C in place to fp16, and the
//               d-scaled copy of X in fp16.  theta, dt and lambda are prefetched
//               into registers one chunk ahead.
//   warps 6-9   epilogue (one thread per TMEM lane): mask the scores in TMEM into
//               bf16 hi/lo pairs (GEMM2 reads them from TMEM), advance the fp32
//               state (kept in registers) and write its scaled fp16 copy for
//               GEMM3, and write y.
// Operand precision: B~, C~, the state copy and d X are fp16 (11 significant
// bits; the state copy carries a per-chunk power-of-two scale), the masked scores
// are bf16 hi + lo (about 16 bits, full fp32 range), X is the exact bf16 input;
// every product accumulates in fp32 in TMEM.  The measured error of this scheme
// is about 0.6-0.8% of the output RMS at the benchmark shapes.
// TMEM (512 columns): [0,256) two score buffers, [256,320) C~H, [320,384) PX,
// [384,448) the chunk's state increment U.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "m3_internal.h"
#include "m3_ptx.cuh"

namespace m3 {
namespace {

constexpr int kRows = 128;  // (token, rank) rows per chunk
constexpr int kP = 64;      // head dimension handled by this kernel
constexpr int kThreads = 320;
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpXf = 2, kWarpEpi = 6;
constexpr int kRole = 128;  // threads of the transform and of the epilogue role
constexpr uint32_t kBarXf = 1, kBarEpi = 2;  // named barrier ids
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_S = 0, TM_YOFF = 256, TM_YIN = 320, TM_U = 384;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTwoPi = 6.283185307179586f;
constexpr float kInvTwoPi = 0.15915494309189535f;
constexpr float kF16Max = 65504.f;

// mbarriers
enum {
  B_FULL = 0,    // [2] TMA tiles of a stage landed
  B_SFREE = 2,   // [2] stage and score buffer free again (commit after GEMM2)
  B_XF = 4,      // [2] transform finished a chunk (4 warp arrivals)
  B_SFULL = 6,   // [2] scores in TMEM (commit after GEMM1)
  B_PFULL = 8,   // [2] masked scores written back (4 warp arrivals)
  B_UFULL = 10,  // state increment U in TMEM (commit after GEMM4)
  B_STATE = 11,  // state advanced: U read, next h^T copy in shared memory (4 arrivals)
  B_HFREE = 12,  // GEMM3 finished reading h^T (commit)
  B_YFULL = 13,  // GEMM2 finished: both output accumulators complete (commit)
  B_YFREE = 14,  // epilogue read both output accumulators (4 arrivals)
  NUM_BARS = 15
};

struct TcParams {
  CUtensorMap tmB;  // B [B][T][H][R][N] bf16, box {64, R, 1, CT, 1}
  CUtensorMap tmC;  // C, same
  CUtensorMap tmX;  // x [B][T][H][R][P] bf16, box {64, R, 1, CT, 1}
  const __nv_bfloat16* x;
  const __nv_bfloat16* B;
  const __nv_bfloat16* dt;
  const __nv_bfloat16* lam;
  const __nv_bfloat16* theta;
  const float* A;
  const float* h0;
  const float* phi0;
  const __nv_bfloat16* prevB0;
  const __nv_bfloat16* prevx0;
  float* hT;
  float* phiT;
  __nv_bfloat16* prevBT;
  __nv_bfloat16* prevxT;
  void* y;
  int out_bf16;
  int T, H;
  unsigned* status;
};

template <int NS, int R>
struct Cfg {
  static constexpr int CT = kRows / R;   // tokens per chunk
  static constexpr int NB = NS / 64;     // 64-wide blocks of the state dimension
  static constexpr int K = NS / 2;       // rotation pairs
  static constexpr int PG = K / 4;       // 16-byte groups (4 pairs) per row
  static constexpr int TB = kRole / PG;  // token blocks of the rotation
  static constexpr int TPT = CT / TB;    // tokens per rotation thread
  static constexpr int kLogR = R == 1 ? 0 : R == 2 ? 1 : R == 4 ? 2 : 3;
  // shared memory (bytes from a 1024-aligned base)
  static constexpr uint32_t TILE = NB * 16384;        // 128 rows x NS, bf16 or fp16
  static constexpr uint32_t STAGE = 2 * TILE + 16384;  // B~, C~, X
  static constexpr uint32_t OFF_DX = 2 * STAGE;        // d X, fp16 [128 rows][64]
  static constexpr uint32_t OFF_H = OFF_DX + 16384;    // h^T, fp16 [NB][64 p][64 n]
  static constexpr uint32_t OFF_MISC = OFF_H + NB * 8192;
  // misc floats
  static constexpr int M_ELL = 0;             // [2][128] decay log2-sums
  static constexpr int M_W = 256;             // [2][128] trapezoid column weights
  static constexpr int M_GAM = 512;           // [2][128] diagonal weights
  static constexpr int M_EL = 768;            // [2][128] 2^{l}
  static constexpr int M_ELAST = 1024;        // [2] 2^{l_last}
  static constexpr int M_D = 1028;            // [128] d_j
  static constexpr int M_DT = 1156;           // [128] dt
  static constexpr int M_Q = 1284;            // [129] q, then q of the next chunk's first token
  static constexpr int M_WSUM = 1416;         // [4] warp totals of the log2-decay scan
  static constexpr int M_HMAX = 1420;         // [2][4] per-warp max |h|
  static constexpr int M_CARRY = 1428;        // [2][64] angle carried into a chunk
  static constexpr int M_SCAN = 1556;         // [TB][K] angle partial sums
  static constexpr int M_END = M_SCAN + TB * K;
  static constexpr uint32_t OFF_BAR = OFF_MISC + ((M_END * 4 + 15) / 16) * 16;
  static constexpr uint32_t OFF_HOLD = OFF_BAR + NUM_BARS * 8;  // TMEM base, abort flag
  static constexpr uint32_t SMEM_USED = OFF_HOLD + 16;
  static constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
  static_assert(kRows % R == 0, "R must divide 128");
  static_assert(NS == 64 || NS == 128, "N must be 64 or 128");
  static_assert(TB * TPT == CT, "token split");
  static_assert(CT <= kRole, "one discretisation thread per token");
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk16) {
  return row * 128u + (((chunk16 ^ (row & 7u)) & 7u) << 4);
}

__device__ __forceinline__ float reduce_angle(float a) {
  return fmaf(-kTwoPi, rintf(a * kInvTwoPi), a);
}

// v = hi + lo with hi = bf16(v) and lo = bf16(v - hi): about 16 significant bits.
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Power of two s with max_abs * s in [2^14, 2^15): the fp16 state copy keeps full
// relative precision and stays far from overflow.  1 for a zero (or denormal) state.
__device__ __forceinline__ float state_scale(float max_abs) {
  const int e = (__float_as_int(max_abs) >> 23) & 0xff;
  if (e == 0) return 1.f;
  int f = 268 - e;  // exponent field of 2^(141 - e)
  f = f < 1 ? 1 : (f > 254 ? 254 : f);
  return __int_as_float(f << 23);
}

template <int NS, int R>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ TcParams p) {
  using C = Cfg<NS, R>;
  constexpr int CT = C::CT, NB = C::NB, K = C::K, PG = C::PG, TB = C::TB, TPT = C::TPT;
  constexpr int KS = NS / 16;  // k-steps over the state dimension

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  float* misc = reinterpret_cast<float*>(sm + C::OFF_MISC);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + C::OFF_HOLD);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + C::OFF_HOLD + 4);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x, b = bh / p.H, head = bh % p.H, H = p.H;
  const int T = p.T;
  const int nchunks = (T + CT - 1) / CT;
  const float A2 = p.A[head] * kLog2e;

  if (tid == 0) {
    const int counts[NUM_BARS] = {1, 1, 1, 1, 4, 4, 1, 1, 4, 4, 1, 4, 1, 1, 4};
    for (int i = 0; i < NUM_BARS; ++i) mbar_init(bar(i), counts[i]);
    *s_abort = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&p.tmB);
    tma_prefetch_desc(&p.tmC);
    tma_prefetch_desc(&p.tmX);
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(s_tmem), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == kWarpTma) {
    // ================================================================ TMA producer
    if (lane == 0) {
      int issued[2] = {-1, -1};
      for (int k = 0; k < nchunks; ++k) {
        const int s = k & 1;
        if (k >= 2 && !mbar_wait_abortable(bar(B_SFREE + s), ((k >> 1) - 1) & 1, s_abort)) break;
        const uint32_t st = sbase + s * C::STAGE;
        mbar_arrive_expect_tx(bar(B_FULL + s), C::STAGE);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          tma_load_5d(st + nb * 16384, &p.tmB, bar(B_FULL + s), 64 * nb, 0, head, k * CT, b);
          tma_load_5d(st + C::TILE + nb * 16384, &p.tmC, bar(B_FULL + s), 64 * nb, 0, head, k * CT, b);
        }
        tma_load_5d(st + 2 * C::TILE, &p.tmX, bar(B_FULL + s), 0, 0, head, k * CT, b);
        issued[s] = k;
      }
      // no copy may still be in flight when the CTA exits
      for (int s = 0; s < 2; ++s)
        if (issued[s] >= 0) mbar_wait(bar(B_FULL + s), (issued[s] >> 1) & 1);
    }
  } else if (warp == kWarpMma) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t I_S = idesc_f16(128, 128, 0, 0);   // S = C~ B~^T
      constexpr uint32_t I_CH = idesc_f16(128, 64, 0, 0);   // Y_off = C~ H
      constexpr uint32_t I_U = idesc_f16(128, 64, 1, 1);    // U = B~^T (d X)
      constexpr uint32_t I_PX = idesc_bf16(128, 64, 0, 1);  // Y_in = P X
      const uint32_t sDX = sbase + C::OFF_DX, sH = sbase + C::OFF_H;
      int last_bar = -1;
      uint32_t last_par = 0;
      for (int k = 0; k < nchunks; ++k) {
        const int s = k & 1;
        const uint32_t st = sbase + s * C::STAGE;
        const uint32_t sB = st, sC = st + C::TILE, sX = st + 2 * C::TILE;
        const uint32_t tS = tmem + TM_S + 128u * s;
        if (!mbar_wait_abortable(bar(B_XF + s), (k >> 1) & 1, s_abort)) break;
        if (k >= 2 && !mbar_wait_abortable(bar(B_SFREE + s), ((k >> 1) - 1) & 1, s_abort)) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const uint32_t ko = (ks >> 2) * 16384u + (ks & 3) * 32u;
          tc_mma_ss(tS, sdesc_sw128(sC + ko, 16, 1024), sdesc_sw128(sB + ko, 16, 1024), I_S, ks > 0);
        }
        tc_commit(bar(B_SFULL + s));
        last_bar = B_SFULL + s;
        last_par = (k >> 1) & 1;
        if (!mbar_wait_abortable(bar(B_STATE), k & 1, s_abort)) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kRows / 16; ++ks) {
          const uint32_t kr = ks * 2048u;
          tc_mma_ss(tmem + TM_U, sdesc_sw128(sB + kr, 16384, 1024), sdesc_sw128(sDX + kr, 16384, 1024),
                    I_U, ks > 0);
        }
        tc_commit(bar(B_UFULL));
        last_bar = B_UFULL;
        last_par = k & 1;
        if (k >= 1 && !mbar_wait_abortable(bar(B_YFREE), (k - 1) & 1, s_abort)) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const uint32_t ka = (ks >> 2) * 16384u + (ks & 3) * 32u;
          const uint32_t kh = (ks >> 2) * 8192u + (ks & 3) * 32u;
          tc_mma_ss(tmem + TM_YOFF, sdesc_sw128(sC + ka, 16, 1024), sdesc_sw128(sH + kh, 16, 1024), I_CH,
                    ks > 0);
        }
        tc_commit(bar(B_HFREE));
        last_bar = B_HFREE;
        last_par = k & 1;
        if (!mbar_wait_abortable(bar(B_PFULL + s), (k >> 1) & 1, s_abort)) break;
        tc_fence_after();
        // masked scores as A from TMEM: per 32-column block, 16 columns of bf16 hi pairs
        // then 16 columns of lo pairs; each MMA takes K = 16 rows of X.
#pragma unroll
        for (int blk = 0; blk < 4; ++blk)
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
              const uint32_t j0 = 32u * blk + 16u * sub;
              tc_mma_ts(tmem + TM_YIN, tS + 32u * blk + 16u * part + 8u * sub,
                        sdesc_sw128(sX + j0 * 128u, 16384, 1024), I_PX, (blk | part | sub) != 0);
            }
        tc_commit(bar(B_YFULL));
        tc_commit(bar(B_SFREE + s));
        last_bar = B_SFREE + s;
        last_par = (k >> 1) & 1;
      }
      // every MMA must be complete before the TMEM is released (the last commit tracks all)
      if (last_bar >= 0) mbar_wait(bar(last_bar), last_par);
    }
  } else if (warp < kWarpEpi) {
    // ================================================================ transform
    const int xt = tid - kWarpXf * 32;  // 0..127
    const int xw = xt >> 5;
    const int pg = xt % PG, tb = xt / PG;
    float* s_ell = misc + C::M_ELL;
    float* s_w = misc + C::M_W;
    float* s_gam = misc + C::M_GAM;
    float* s_el = misc + C::M_EL;
    float* s_elast = misc + C::M_ELAST;
    float* s_d = misc + C::M_D;
    float* s_dt = misc + C::M_DT;
    float* s_q = misc + C::M_Q;
    float* s_wsum = misc + C::M_WSUM;
    float* s_carry = misc + C::M_CARRY;
    float* s_scan = misc + C::M_SCAN;
    const size_t tok_stride = static_cast<size_t>(H);
    const size_t seq0 = static_cast<size_t>(b) * T * H + head;  // token 0 of this sequence

    auto load_tok = [&](int kk, float& d, float& l) {
      const int t = kk * CT + xt;
      d = 0.f;
      l = 0.f;
      if (xt < CT && t < T) {
        d = __bfloat162float(p.dt[seq0 + t * tok_stride]);
        l = __bfloat162float(p.lam[seq0 + t * tok_stride]);
      }
    };
    auto load_q = [&](int kk) -> float {
      const int t = kk * CT;
      if (xt != 0 || t >= T) return 0.f;
      return (1.f - __bfloat162float(p.lam[seq0 + t * tok_stride])) *
             __bfloat162float(p.dt[seq0 + t * tok_stride]);
    };
    auto load_th = [&](int kk, uint2 (&th)[TPT]) {
#pragma unroll
      for (int u = 0; u < TPT; ++u) {
        const int t = kk * CT + tb * TPT + u;
        th[u] = make_uint2(0u, 0u);
        if (t < T)
          th[u] = *reinterpret_cast<const uint2*>(p.theta + (seq0 + t * tok_stride) * K + 4 * pg);
      }
    };

    float cur_dt, cur_lam, nxt_dt = 0.f, nxt_lam = 0.f;
    uint2 th_cur[TPT], th_nxt[TPT];
    load_tok(0, cur_dt, cur_lam);
    float qn_cur = load_q(1), qn_nxt = 0.f;
    load_th(0, th_cur);
#pragma unroll
    for (int u = 0; u < TPT; ++u) th_nxt[u] = make_uint2(0u, 0u);
    for (int k = xt; k < K; k += kRole) s_carry[k] = reduce_angle(p.phi0 ? p.phi0[static_cast<size_t>(bh) * K + k] : 0.f);
    float range = 0.f;  // largest |value| converted to fp16
    bool ab = false;

    for (int k = 0; k < nchunks; ++k) {
      const int s = k & 1;
      if (k + 1 < nchunks) {
        load_tok(k + 1, nxt_dt, nxt_lam);
        load_th(k + 1, th_nxt);
      }
      qn_nxt = load_q(k + 2);
      // ---------------------------------------------------------- step A: decay scan
      const float a2 = cur_dt * A2;
      const float gam = cur_lam * cur_dt;
      float incl = a2;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (lane == 31) s_wsum[xw] = incl;
      if (xt < CT) {
        s_q[xt] = (1.f - cur_lam) * cur_dt;
        s_dt[xt] = cur_dt;
      }
      if (xt == 0) s_q[CT] = qn_cur;
      // the epilogue must be done with this misc slot (chunk k - 2)
      if (k >= 2) ab = ab || !__all_sync(0xffffffffu, mbar_wait_abortable(bar(B_PFULL + s), ((k >> 1) - 1) & 1, s_abort));
      if (bar_sync_or(kBarXf, kRole, ab)) { ab = true; break; }
      // ---------------------------------------------------------- step B: weights, angle partials
      {
        float ell = incl, ltot = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float v = s_wsum[w];
          ltot += v;
          if (w < xw) ell += v;
        }
        if (xt < CT) {
          const float w = gam + s_q[xt + 1];
          s_ell[s * 128 + xt] = ell;
          s_w[s * 128 + xt] = w;
          s_gam[s * 128 + xt] = gam;
          s_el[s * 128 + xt] = ex2(ell);
          s_d[xt] = ex2(ltot - ell) * w;
        }
        if (xt == 0) s_elast[s] = ex2(ltot);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int u = 0; u < TPT; ++u) {
          const float d = s_dt[tb * TPT + u];
          const float2 t01 = unpack_bf16x2(th_cur[u].x), t23 = unpack_bf16x2(th_cur[u].y);
          acc[0] = fmaf(d, t01.x, acc[0]);
          acc[1] = fmaf(d, t01.y, acc[1]);
          acc[2] = fmaf(d, t23.x, acc[2]);
          acc[3] = fmaf(d, t23.y, acc[3]);
        }
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) s_scan[tb * K + 4 * pg + qq] = acc[qq];
      }
      if (bar_sync_or(kBarXf, kRole, ab)) { ab = true; break; }
      // ---------------------------------------------------------- step C: rotate B, C; d X
      {
        float ang[4];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) ang[qq] = s_carry[s * 64 + 4 * pg + qq];
        for (int t2 = 0; t2 < tb; ++t2)
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) ang[qq] += s_scan[t2 * K + 4 * pg + qq];
        ab = ab || !__all_sync(0xffffffffu, mbar_wait_abortable(bar(B_FULL + s), (k >> 1) & 1, s_abort));
        if (!ab) {
          uint8_t* stg = sm + s * C::STAGE;
          const int nb = pg >> 3, c16 = pg & 7;
#pragma unroll
          for (int u = 0; u < TPT; ++u) {
            const float d = s_dt[tb * TPT + u];
            const float2 t01 = unpack_bf16x2(th_cur[u].x), t23 = unpack_bf16x2(th_cur[u].y);
            ang[0] = fmaf(d, t01.x, ang[0]);
            ang[1] = fmaf(d, t01.y, ang[1]);
            ang[2] = fmaf(d, t23.x, ang[2]);
            ang[3] = fmaf(d, t23.y, ang[3]);
            float cs[4], sn[4];
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) __sincosf(reduce_angle(ang[qq]), &sn[qq], &cs[qq]);
            const int i = tb * TPT + u;
#pragma unroll
            for (int r = 0; r < R; ++r) {
              const uint32_t off = nb * 16384u + sw128(i * R + r, c16);
              uint4 vb = *reinterpret_cast<const uint4*>(stg + off);
              uint4 vc = *reinterpret_cast<const uint4*>(stg + C::TILE + off);
              uint32_t* wb = reinterpret_cast<uint32_t*>(&vb);
              uint32_t* wc = reinterpret_cast<uint32_t*>(&vc);
#pragma unroll
              for (int qq = 0; qq < 4; ++qq) {
                const float2 bb = unpack_bf16x2(wb[qq]), cc = unpack_bf16x2(wc[qq]);
                const float b0 = cs[qq] * bb.x + sn[qq] * bb.y, b1 = -sn[qq] * bb.x + cs[qq] * bb.y;
                const float c0 = cs[qq] * cc.x + sn[qq] * cc.y, c1 = -sn[qq] * cc.x + cs[qq] * cc.y;
                range = fmaxf(range, fmaxf(fmaxf(fabsf(b0), fabsf(b1)), fmaxf(fabsf(c0), fabsf(c1))));
                wb[qq] = pack_f16x2(b0, b1);
                wc[qq] = pack_f16x2(c0, c1);
              }
              *reinterpret_cast<uint4*>(stg + off) = vb;
              *reinterpret_cast<uint4*>(stg + C::TILE + off) = vc;
            }
          }
          if (tb == TB - 1) {
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) s_carry[(s ^ 1) * 64 + 4 * pg + qq] = reduce_angle(ang[qq]);
          }
        }
        // d X into the single fp16 buffer, once GEMM4 of the previous chunk has read it
        if (k >= 1) ab = ab || !__all_sync(0xffffffffu, mbar_wait_abortable(bar(B_UFULL), (k - 1) & 1, s_abort));
        if (!ab) {
          const uint8_t* sx = sm + s * C::STAGE + 2 * C::TILE;
          uint8_t* sdx = sm + C::OFF_DX;
          const float dv = s_d[xt >> C::kLogR];
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const uint32_t off = sw128(xt, g);
            uint4 v = *reinterpret_cast<const uint4*>(sx + off);
            uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              const float2 xx = unpack_bf16x2(w[qq]);
              const float a0 = dv * xx.x, a1 = dv * xx.y;
              range = fmaxf(range, fmaxf(fabsf(a0), fabsf(a1)));
              w[qq] = pack_f16x2(a0, a1);
            }
            *reinterpret_cast<uint4*>(sdx + off) = v;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_XF + s));
        }
      }
      cur_dt = nxt_dt;
      cur_lam = nxt_lam;
      qn_cur = qn_nxt;
#pragma unroll
      for (int u = 0; u < TPT; ++u) th_cur[u] = th_nxt[u];
    }
    if (range > kF16Max) atomicOr(p.status, kDevRange);
    // ---------------------------------------------------------------- exit angle and token
    bar_sync_or(kBarXf, kRole, ab);
    if (!ab) {
      if (p.phiT)
        for (int k = xt; k < K; k += kRole)
          p.phiT[static_cast<size_t>(bh) * K + k] = s_carry[(nchunks & 1) * 64 + k];
      const size_t last = (seq0 + static_cast<size_t>(T - 1) * tok_stride);
      if (p.prevBT)
        for (int e = xt; e < R * NS; e += kRole)
          p.prevBT[static_cast<size_t>(bh) * R * NS + e] = p.B[last * R * NS + e];
      if (p.prevxT)
        for (int e = xt; e < R * kP; e += kRole)
          p.prevxT[static_cast<size_t>(bh) * R * kP + e] = p.x[last * R * kP + e];
    }
  } else {
    // ================================================================ epilogue
    const int q = warp & 3;          // TMEM lane quarter of this warp
    const int ew = warp - kWarpEpi;  // epilogue warp index 0..3
    const int i = q * 32 + lane;     // TMEM lane = chunk row = state row
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const bool srow = i < NS;
    const float* s_ell = misc + C::M_ELL;
    const float* s_w = misc + C::M_W;
    const float* s_gam = misc + C::M_GAM;
    const float* s_el = misc + C::M_EL;
    const float* s_elast = misc + C::M_ELAST;
    float* s_hmax = misc + C::M_HMAX;
    uint8_t* sHb = sm + C::OFF_H;
    const size_t seq0 = static_cast<size_t>(b) * T * H + head;

    float hv[kP];
    // -------------------------------------------------------------- entry state
    // H' = h0 + q_0 B~_{-1} X_{-1}^T: the stored previous token rotated by its own angle
    // phi0, weighted by q_0 = (1 - lambda_0) dt_0 of this call's first token.
    {
      const float q0 = (1.f - __bfloat162float(p.lam[seq0])) * __bfloat162float(p.dt[seq0]);
      float bt[R];
#pragma unroll
      for (int r = 0; r < R; ++r) bt[r] = 0.f;
      if (srow && p.prevB0) {
        const int kk = i >> 1;
        const float ph = p.phi0 ? p.phi0[static_cast<size_t>(bh) * K + kk] : 0.f;
        float sn, cs;
        sincosf(ph, &sn, &cs);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const __nv_bfloat16* pb = p.prevB0 + (static_cast<size_t>(bh) * R + r) * NS + 2 * kk;
          const float u = __bfloat162float(pb[0]), v = __bfloat162float(pb[1]);
          bt[r] = (i & 1) ? (-sn * u + cs * v) : (cs * u + sn * v);
        }
      }
#pragma unroll
      for (int pp = 0; pp < kP; ++pp) {
        float v = 0.f;
        if (srow) {
          if (p.h0) v = p.h0[(static_cast<size_t>(bh) * NS + i) * kP + pp];
          if (p.prevx0) {
            float f = 0.f;
#pragma unroll
            for (int r = 0; r < R; ++r)
              f = fmaf(bt[r], __bfloat162float(p.prevx0[(static_cast<size_t>(bh) * R + r) * kP + pp]), f);
            v = fmaf(q0, f, v);
          }
        }
        hv[pp] = v;
      }
    }
    // Scaled fp16 copy of the state as the K-major B operand of GEMM3 (row p, column n).
    auto put_state = [&](float sig) {
      if (srow) {
        const uint32_t base = (i >> 6) * 8192u + (i & 7) * 2;
#pragma unroll
        for (int pp = 0; pp < kP; ++pp)
          *reinterpret_cast<__half*>(sHb + base + sw128(pp, (i & 63) >> 3)) = __float2half_rn(sig * hv[pp]);
      }
    };
    auto max_abs = [&]() {
      float mx = 0.f;
#pragma unroll
      for (int pp = 0; pp < kP; ++pp) mx = fmaxf(mx, fabsf(hv[pp]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      return mx;
    };
    bool ab = false;
    float sig_cur;
    {
      const float mx = max_abs();
      if (lane == 0) s_hmax[ew] = mx;
      bar_sync_or(kBarEpi, kRole, false);
      sig_cur = state_scale(fmaxf(fmaxf(s_hmax[0], s_hmax[1]), fmaxf(s_hmax[2], s_hmax[3])));
      put_state(sig_cur);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_STATE));
    }

    for (int k = 0; k < nchunks; ++k) {
      const int s = k & 1;
      const int t0 = k * CT;
      const uint32_t tS = tmem + TM_S + 128u * s;
      const int ti = i >> C::kLogR;
      // ---------------------------------------------------------- mask: S -> P (bf16 hi/lo)
      // (the transform's arrival on B_XF publishes this chunk's decay sums and weights)
      ab = ab || !__all_sync(0xffffffffu, mbar_wait_abortable(bar(B_XF + s), (k >> 1) & 1, s_abort));
      ab = ab || !__all_sync(0xffffffffu, mbar_wait_abortable(bar(B_SFULL + s), (k >> 1) & 1, s_abort));
      const float el_i = ab ? 0.f : s_el[s * 128 + ti];
      if (!ab) {
        tc_fence_after();
        const float ell_i = s_ell[s * 128 + ti], gam_i = s_gam[s * 128 + ti];
        const int whi = (q * 32 + 31) >> C::kLogR;  // last token among this warp's rows
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          uint32_t hi[16], lo[16];
          if (((32 * blk) >> C::kLogR) > whi) {
#pragma unroll
            for (int c = 0; c < 16; ++c) hi[c] = lo[c] = 0u;
          } else {
            uint32_t sv[32];
            tmem_ld32(tS + lane_off + 32u * blk, sv);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              float m2[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int tj = (32 * blk + c + e) >> C::kLogR;
                float m = 0.f;
                if (tj < ti) m = ex2(ell_i - s_ell[s * 128 + tj]) * s_w[s * 128 + tj];
                else if (tj == ti) m = gam_i;
                m2[e] = m * __uint_as_float(sv[c + e]);
              }
              split2(m2[0], m2[1], hi[c >> 1], lo[c >> 1]);
            }
          }
          tmem_st16(tS + lane_off + 32u * blk, hi);
          tmem_st16(tS + lane_off + 32u * blk + 16u, lo);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PFULL + s));
      }
      // ---------------------------------------------------------- state: H <- e^{L} H + U
      ab = ab || !__all_sync(0xffffffffu, mbar_wait_abortable(bar(B_UFULL), k & 1, s_abort));
      ab = ab || !__all_sync(0xffffffffu, mbar_wait_abortable(bar(B_HFREE), k & 1, s_abort));
      float mx = 0.f;
      if (!ab) {
        tc_fence_after();
        if (q * 32 < NS) {  // warp-uniform: this warp owns state rows
          const float eL = s_elast[s];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t uv[32];
            tmem_ld32(tmem + TM_U + lane_off + 32u * half, uv);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) hv[32 * half + j] = fmaf(eL, hv[32 * half + j], __uint_as_float(uv[j]));
          }
        }
        mx = max_abs();
        if (lane == 0) s_hmax[(s ^ 1) * 4 + ew] = mx;
      }
      if (bar_sync_or(kBarEpi, kRole, ab)) { ab = true; break; }
      const float sig_next = state_scale(fmaxf(fmaxf(s_hmax[(s ^ 1) * 4 + 0], s_hmax[(s ^ 1) * 4 + 1]),
                                               fmaxf(s_hmax[(s ^ 1) * 4 + 2], s_hmax[(s ^ 1) * 4 + 3])));
      put_state(sig_next);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_STATE));
      // ---------------------------------------------------------- y = P X + e^{l} C~ H
      ab = ab || !__all_sync(0xffffffffu, mbar_wait_abortable(bar(B_YFULL), k & 1, s_abort));
      if (!ab) {
        tc_fence_after();
        const float f = el_i / sig_cur;
        const int r = i & (R - 1);
        const int t = t0 + ti;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t a[32], c[32];
          tmem_ld32(tmem + TM_YIN + lane_off + 32u * half, a);
          tmem_ld32(tmem + TM_YOFF + lane_off + 32u * half, c);
          tmem_ld_wait();
          if (t < T) {
            const size_t o = ((seq0 + static_cast<size_t>(t) * H) * R + r) * kP + 32 * half;
            if (p.out_bf16) {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.y) + o);
#pragma unroll
              for (int qq = 0; qq < 4; ++qq) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int j = 8 * qq + 2 * e;
                  w[e] = pack_bf16x2(fmaf(f, __uint_as_float(c[j]), __uint_as_float(a[j])),
                                     fmaf(f, __uint_as_float(c[j + 1]), __uint_as_float(a[j + 1])));
                }
                dst[qq] = make_uint4(w[0], w[1], w[2], w[3]);
              }
            } else {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.y) + o);
#pragma unroll
              for (int qq = 0; qq < 8; ++qq) {
                float v[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  v[e] = fmaf(f, __uint_as_float(c[4 * qq + e]), __uint_as_float(a[4 * qq + e]));
                dst[qq] = make_float4(v[0], v[1], v[2], v[3]);
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_YFREE));
      }
      sig_cur = sig_next;
    }
    // ---------------------------------------------------------------- exit state
    if (!ab && p.hT && srow) {
      float4* dst = reinterpret_cast<float4*>(p.hT + (static_cast<size_t>(bh) * NS + i) * kP);
#pragma unroll
      for (int qq = 0; qq < kP / 4; ++qq)
        dst[qq] = make_float4(hv[4 * qq], hv[4 * qq + 1], hv[4 * qq + 2], hv[4 * qq + 3]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0 && *s_abort) atomicOr(p.status, kDevTimeout);
  if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 5-D map over [B][T][H][R][inner] bf16 with a box of {64, R, 1, ct, 1}.
bool make_map(CUtensorMap* m, const void* ptr, int Bsz, int T, int H, int R, int inner, int ct) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[5] = {(cuuint64_t)inner, (cuuint64_t)R, (cuuint64_t)H, (cuuint64_t)T,
                              (cuuint64_t)Bsz};
  const cuuint64_t e = 2;
  const cuuint64_t strides[4] = {e * inner, e * inner * R, e * inner * R * H,
                                 e * inner * R * H * (cuuint64_t)T};
  const cuuint32_t box[5] = {64u, (cuuint32_t)R, 1u, (cuuint32_t)ct, 1u};
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(ptr), dims, strides, box,
                  es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int NS, int R>
cudaError_t launch_nr(const PrefillArgs& a, cudaStream_t s) {
  using C = Cfg<NS, R>;
  const m3_dims& d = a.d;
  TcParams p;
  if (!make_map(&p.tmB, a.B, d.B, d.T, d.H, R, NS, C::CT) ||
      !make_map(&p.tmC, a.C, d.B, d.T, d.H, R, NS, C::CT) ||
      !make_map(&p.tmX, a.x, d.B, d.T, d.H, R, kP, C::CT))
    return cudaErrorInvalidValue;
  p.x = static_cast<const __nv_bfloat16*>(a.x);
  p.B = static_cast<const __nv_bfloat16*>(a.B);
  p.dt = static_cast<const __nv_bfloat16*>(a.dt);
  p.lam = static_cast<const __nv_bfloat16*>(a.lam);
  p.theta = static_cast<const __nv_bfloat16*>(a.theta);
  p.A = a.A;
  p.h0 = a.h0.h;
  p.phi0 = a.h0.phi;
  p.prevB0 = static_cast<const __nv_bfloat16*>(a.h0.prev_B);
  p.prevx0 = static_cast<const __nv_bfloat16*>(a.h0.prev_x);
  p.hT = a.hT.h;
  p.phiT = a.hT.phi;
  p.prevBT = static_cast<__nv_bfloat16*>(a.hT.prev_B);
  p.prevxT = static_cast<__nv_bfloat16*>(a.hT.prev_x);
  p.y = a.y;
  p.out_bf16 = d.out_dtype == M3_BF16;
  p.T = d.T;
  p.H = d.H;
  p.status = a.status;
  auto k = prefill_tc_kernel<NS, R>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  k<<<static_cast<unsigned>(d.B) * static_cast<unsigned>(d.H), kThreads, C::SMEM_ALLOC, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(const m3_dims& d) {
  return d.in_dtype == M3_BF16 && d.P == kP && (d.N == 64 || d.N == 128) &&
         (d.R == 1 || d.R == 2 || d.R == 4 || d.R == 8) && (d.chunk == 0 || d.chunk == kRows / d.R);
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s) {
#define M3_NR(NN, RR) \
  if (a.d.N == NN && a.d.R == RR) return launch_nr<NN, RR>(a, s);
  M3_NR(128, 1)
  M3_NR(128, 2)
  M3_NR(128, 4)
  M3_NR(128, 8)
  M3_NR(64, 1)
  M3_NR(64, 2)
  M3_NR(64, 4)
  M3_NR(64, 8)
#undef M3_NR
  return cudaErrorInvalidValue;
}

}  // namespace m3
