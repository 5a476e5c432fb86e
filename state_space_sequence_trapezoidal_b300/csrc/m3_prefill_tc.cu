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
//     S = C~ B~^T                                  (GEMM1, 128 x 128 x N)
//     Y = (M (x) J_R o S) X + diag(e^{l}) C~ H     (GEMM2, GEMM3)
//     H <- e^{l_last} H + B~^T diag(d) X,  d_j = e^{l_last - l_j} w_j   (GEMM4)
// where w of the chunk's last token takes q of the next chunk's first token,
// which carries the trapezoid's previous-token term across the boundary.
//
// Kernel design (one CTA per (batch row, head), two CTAs per SM, 256 threads):
//  * B, C, X tiles of 128 rows arrive by TMA (128-byte swizzle, zero fill past T).
//  * All threads rotate B and C in place in shared memory by the cumulative angle
//    (a prefix sum over the chunk plus the carried angle), Proposition 3.
//  * One thread issues the four GEMMs (tcgen05.mma kind::f16, bf16 operands,
//    fp32 accumulators in TMEM).  The mask is applied between GEMM1 and GEMM2 by
//    all eight warps reading S from TMEM.  The fp32 state H stays in TMEM across
//    the whole sequence; a bf16 copy in shared memory feeds GEMM3.
//  * Decay factors are kept as log2 sums and only non-positive differences are
//    exponentiated, so nothing overflows however long the chunk.
// TMEM (256 columns): [0,128) S, later U = B~^T diag(d) X in [0,64);
//                     [128,192) Y; [192,256) H (fp32, N lanes x 64 columns).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "m3_internal.h"
#include "m3_ptx.cuh"

namespace m3 {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 128;         // (token, rank) rows per chunk
constexpr int kP = 64;             // head dimension handled by this kernel
constexpr uint32_t kTmemCols = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTwoPi = 6.283185307179586f;
constexpr float kInvTwoPi = 0.15915494309189535f;

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
  static constexpr int CT = kRows / R;               // tokens per chunk
  static constexpr int NB = NS / 64;                 // 64-wide blocks of the state dim
  static constexpr int K = NS / 2;                   // rotation pairs
  static constexpr int PG = K / 4;                   // 16-byte groups (4 pairs) per row
  static constexpr int TB = (kThreads / PG < CT) ? kThreads / PG : CT;  // token blocks
  static constexpr int TPT = CT / TB;                // tokens per rotation thread
  static constexpr int kLogR = R == 1 ? 0 : R == 2 ? 1 : R == 4 ? 2 : 3;
  // Shared memory map (bytes from a 1024-aligned base).  Every rounded GEMM operand is
  // held as a bf16 pair (hi, lo) with hi = bf16(v), lo = bf16(v - hi).
  static constexpr uint32_t TILE = NB * 16384;        // one 128-row tile of width NS
  static constexpr uint32_t OFF_B = 0;                // B~ hi   [NB][128 rows][128 B]
  static constexpr uint32_t OFF_C = OFF_B + TILE;     // C~ hi
  static constexpr uint32_t OFF_BL = OFF_C + TILE;    // B~ lo
  static constexpr uint32_t OFF_CL = OFF_BL + TILE;   // C~ lo
  static constexpr uint32_t OFF_X = OFF_CL + TILE;    // X (exact bf16)
  static constexpr uint32_t OFF_H = OFF_X + 16384;    // state hi  [NB][64 p][128 B]
  static constexpr uint32_t OFF_HL = OFF_H + NB * 8192;  // state lo
  static constexpr uint32_t OFF_P = OFF_B;            // masked scores hi (32 KB: B, and C if NB == 1)
  static constexpr uint32_t OFF_PL = OFF_BL;          // masked scores lo
  static constexpr uint32_t OFF_MISC = OFF_HL + NB * 8192;
  // misc (floats)
  static constexpr int M_DT = 0;
  static constexpr int M_ELL = M_DT + CT;
  static constexpr int M_GAM = M_ELL + CT;
  static constexpr int M_WGT = M_GAM + CT;
  static constexpr int M_DSC = M_WGT + CT;
  static constexpr int M_EL = M_DSC + CT;
  static constexpr int M_Q = M_EL + CT;               // CT + 1 entries
  static constexpr int M_SCAL = M_Q + CT + 4;         // [0] e^{l_last}
  static constexpr int M_CARRY = M_SCAL + 4;          // [2][64]
  static constexpr int M_SCAN = M_CARRY + 2 * 64;     // [TB][K], also [R][NS] + [R][64] at entry
  static constexpr int SCAN_FLOATS = (TB * K > R * NS + R * 64) ? TB * K : R * NS + R * 64;
  static constexpr int M_END = M_SCAN + SCAN_FLOATS;
  static constexpr uint32_t OFF_BAR = OFF_MISC + ((M_END * 4 + 15) / 16) * 16;
  static constexpr uint32_t SMEM_USED = OFF_BAR + 32;
  static constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
  static_assert(kRows % R == 0, "R must divide 128");
  static_assert(NS == 64 || NS == 128, "N must be 64 or 128");
  static_assert(TB * TPT == CT, "token split");
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

__device__ __forceinline__ void store_split_bf16(uint8_t* hi_base, uint8_t* lo_base, uint32_t off,
                                                 float v) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  *reinterpret_cast<__nv_bfloat16*>(hi_base + off) = h;
  *reinterpret_cast<__nv_bfloat16*>(lo_base + off) = __float2bfloat16_rn(v - __bfloat162float(h));
}

template <int NS, int R>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ TcParams p) {
  using C = Cfg<NS, R>;
  constexpr int CT = C::CT, NB = C::NB, K = C::K, PG = C::PG, TB = C::TB, TPT = C::TPT;
  constexpr int KS = NS / 16;  // k-steps over the state dimension

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  const uint32_t sB = sbase + C::OFF_B, sC = sbase + C::OFF_C, sBl = sbase + C::OFF_BL,
                 sCl = sbase + C::OFF_CL, sX = sbase + C::OFF_X, sH = sbase + C::OFF_H,
                 sHl = sbase + C::OFF_HL, sP = sbase + C::OFF_P, sPl = sbase + C::OFF_PL;
  float* misc = reinterpret_cast<float*>(sm + C::OFF_MISC);
  float* s_dt = misc + C::M_DT;
  float* s_ell = misc + C::M_ELL;
  float* s_gam = misc + C::M_GAM;
  float* s_wgt = misc + C::M_WGT;
  float* s_dsc = misc + C::M_DSC;
  float* s_eL = misc + C::M_EL;
  float* s_q = misc + C::M_Q;
  float* s_scal = misc + C::M_SCAL;
  float* s_carry = misc + C::M_CARRY;
  float* s_scan = misc + C::M_SCAN;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + C::OFF_BAR + 16);
  const uint32_t bar_tma = smem_u32(&bars[0]), bar_mma = smem_u32(&bars[1]);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x, b = bh / p.H, head = bh % p.H, H = p.H;
  const int T = p.T;
  const int nchunks = (T + CT - 1) / CT;
  const float A2 = p.A[head] * kLog2e;

  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&p.tmB);
    tma_prefetch_desc(&p.tmC);
    tma_prefetch_desc(&p.tmX);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(s_tmem), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t tS = tmem, tU = tmem, tY = tmem + 128, tHc = tmem + 192;
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const int trow = (warp & 3) * 32 + lane;  // TMEM lane / tile row owned by this thread
  const int half = warp >> 2;               // which half of the columns

  auto issue_tma = [&](int ck) {
    mbar_arrive_expect_tx(bar_tma, (2 * NB + 1) * 16384);
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      tma_load_5d(sB + nb * 16384, &p.tmB, bar_tma, 64 * nb, 0, head, ck * CT, b);
      tma_load_5d(sC + nb * 16384, &p.tmC, bar_tma, 64 * nb, 0, head, ck * CT, b);
    }
    tma_load_5d(sX, &p.tmX, bar_tma, 0, 0, head, ck * CT, b);
  };
  if (tid == 0 && nchunks > 0) issue_tma(0);

  // Writes H (fp32) of state row n, columns 32*half .. +31, into TMEM and its hi/lo copy
  // into the K-major B operand of GEMM3 (row p, column n of [NB][64][128 B]).
  auto put_state = [&](uint32_t (&hv)[32]) {
    const int n = trow;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int pc = 32 * half + j;
      const uint32_t off = (n >> 6) * 8192u + sw128(pc, (n & 63) >> 3) + (n & 7) * 2;
      store_split_bf16(sm + C::OFF_H, sm + C::OFF_HL, off, __uint_as_float(hv[j]));
    }
    tmem_st32(tHc + lane_off + 32 * half, hv);
    tmem_st_wait();
  };

  // ---------------------------------------------------------------- entry state
  // H' = h0 + q_0 B~_{-1} X_{-1}^T, with B~_{-1} the stored previous token rotated by
  // its own angle phi0 and q_0 = (1 - lambda_0) dt_0 of this call's first token.
  {
    float* s_fb = s_scan;            // [R][NS]
    float* s_fx = s_scan + R * NS;   // [R][64]
    for (int k = tid; k < K; k += kThreads) {
      const float ph = p.phi0 ? p.phi0[static_cast<size_t>(bh) * K + k] : 0.f;
      s_carry[k] = reduce_angle(ph);
      float s, c;
      sincosf(ph, &s, &c);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float u = 0.f, v = 0.f;
        if (p.prevB0) {
          const __nv_bfloat16* pb = p.prevB0 + (static_cast<size_t>(bh) * R + r) * NS + 2 * k;
          u = __bfloat162float(pb[0]);
          v = __bfloat162float(pb[1]);
        }
        s_fb[r * NS + 2 * k] = c * u + s * v;
        s_fb[r * NS + 2 * k + 1] = -s * u + c * v;
      }
    }
    for (int i = tid; i < R * kP; i += kThreads)
      s_fx[i] = p.prevx0 ? __bfloat162float(p.prevx0[static_cast<size_t>(bh) * R * kP + i]) : 0.f;
    __syncthreads();
    float q0 = 0.f;
    if (T > 0) {
      const size_t o = static_cast<size_t>(b) * T * H + head;  // token 0
      const float d0 = __bfloat162float(p.dt[o]), l0 = __bfloat162float(p.lam[o]);
      q0 = (1.f - l0) * d0;
    }
    if ((warp & 3) * 32 < NS) {  // warp-uniform: this warp owns state rows
      const int n = trow;
      uint32_t hv[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int pc = 32 * half + j;
        float v = p.h0 ? p.h0[(static_cast<size_t>(bh) * NS + n) * kP + pc] : 0.f;
        float f = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) f = fmaf(s_fb[r * NS + n], s_fx[r * kP + pc], f);
        hv[j] = __float_as_uint(fmaf(q0, f, v));
      }
      put_state(hv);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
  }

  // Instruction descriptors (M = 128 rows throughout).
  constexpr uint32_t I_S = idesc_bf16(128, 128, 0, 0);  // S = C~ B~^T
  constexpr uint32_t I_CH = idesc_bf16(128, 64, 0, 0);  // Y = C~ H
  constexpr uint32_t I_U = idesc_bf16(128, 64, 1, 1);   // U = B~^T X  (both MN-major)
  constexpr uint32_t I_PX = idesc_bf16(128, 64, 0, 1);  // Y += P X   (X MN-major)

  uint32_t mma_count = 0;
  bool ok = true;

  const bool rot_thread = tid < PG * TB;
  const int pg = tid % PG, tb = tid / PG;

  for (int ck = 0; ck < nchunks; ++ck) {
    const int t0 = ck * CT;
    // ------------------------------------------------------------ discretisation
    if (warp == 0) {
      constexpr int TPL = (CT + 31) / 32;
      float a2[TPL], gm[TPL], qq[TPL];
      float run = 0.f;
#pragma unroll
      for (int u = 0; u < TPL; ++u) {
        const int i = lane * TPL + u;
        const int t = t0 + i;
        float d = 0.f, l = 0.f;
        if (i < CT && t < T) {
          const size_t o = (static_cast<size_t>(b) * T + t) * H + head;
          d = __bfloat162float(p.dt[o]);
          l = __bfloat162float(p.lam[o]);
        }
        run += d * A2;
        a2[u] = run;
        gm[u] = l * d;
        qq[u] = (1.f - l) * d;
        if (i < CT) s_dt[i] = d;
      }
      float incl = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const float excl = incl - run;
#pragma unroll
      for (int u = 0; u < TPL; ++u) {
        const int i = lane * TPL + u;
        if (i < CT) {
          s_ell[i] = excl + a2[u];
          s_gam[i] = gm[u];
          s_q[i] = qq[u];
        }
      }
      if (lane == 0) {
        const int t = t0 + CT;
        float qn = 0.f;
        if (t < T) {
          const size_t o = (static_cast<size_t>(b) * T + t) * H + head;
          qn = (1.f - __bfloat162float(p.lam[o])) * __bfloat162float(p.dt[o]);
        }
        s_q[CT] = qn;
      }
      __syncwarp();
      const float ell_last = s_ell[CT - 1];
#pragma unroll
      for (int u = 0; u < TPL; ++u) {
        const int i = lane * TPL + u;
        if (i < CT) {
          const float w = s_gam[i] + s_q[i + 1];
          s_wgt[i] = w;
          s_dsc[i] = ex2(ell_last - s_ell[i]) * w;
          s_eL[i] = ex2(s_ell[i]);
        }
      }
      if (lane == 0) s_scal[0] = ex2(ell_last);
    }
    // theta for this thread's tokens and pairs (registers)
    float th[TPT][4];
    if (rot_thread) {
#pragma unroll
      for (int u = 0; u < TPT; ++u) {
        const int t = t0 + tb * TPT + u;
        if (t < T) {
          const uint2 raw = *reinterpret_cast<const uint2*>(
              p.theta + ((static_cast<size_t>(b) * T + t) * H + head) * K + 4 * pg);
          const float2 a = unpack_bf16x2(raw.x), c = unpack_bf16x2(raw.y);
          th[u][0] = a.x; th[u][1] = a.y; th[u][2] = c.x; th[u][3] = c.y;
        } else {
          th[u][0] = th[u][1] = th[u][2] = th[u][3] = 0.f;
        }
      }
    }
    __syncthreads();

    // ------------------------------------------------------------ cumulative angle, rotation
    float phl[TPT][4];
    if (rot_thread) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int u = 0; u < TPT; ++u) {
        const float d = s_dt[tb * TPT + u];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[q] = fmaf(d, th[u][q], acc[q]);
          phl[u][q] = acc[q];
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) s_scan[tb * K + 4 * pg + q] = acc[q];
    }
    __syncthreads();
    ok = mbar_wait(bar_tma, ck & 1) && ok;
    if (rot_thread) {
      float base[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) base[q] = s_carry[(ck & 1) * 64 + 4 * pg + q];
      for (int tb2 = 0; tb2 < tb; ++tb2)
#pragma unroll
        for (int q = 0; q < 4; ++q) base[q] += s_scan[tb2 * K + 4 * pg + q];
      const int nb = pg >> 3, c16 = pg & 7;
#pragma unroll
      for (int u = 0; u < TPT; ++u) {
        float cs[4], sn[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) __sincosf(reduce_angle(base[q] + phl[u][q]), &sn[q], &cs[q]);
        const int i = tb * TPT + u;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint32_t off = nb * 16384u + sw128(i * R + r, c16);
          uint4 vb = *reinterpret_cast<const uint4*>(sm + C::OFF_B + off);
          uint4 vc = *reinterpret_cast<const uint4*>(sm + C::OFF_C + off);
          uint4 lb, lc;
          uint32_t* wb = reinterpret_cast<uint32_t*>(&vb);
          uint32_t* wc = reinterpret_cast<uint32_t*>(&vc);
          uint32_t* wlb = reinterpret_cast<uint32_t*>(&lb);
          uint32_t* wlc = reinterpret_cast<uint32_t*>(&lc);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 bb = unpack_bf16x2(wb[q]), cc = unpack_bf16x2(wc[q]);
            split2(cs[q] * bb.x + sn[q] * bb.y, -sn[q] * bb.x + cs[q] * bb.y, wb[q], wlb[q]);
            split2(cs[q] * cc.x + sn[q] * cc.y, -sn[q] * cc.x + cs[q] * cc.y, wc[q], wlc[q]);
          }
          *reinterpret_cast<uint4*>(sm + C::OFF_B + off) = vb;
          *reinterpret_cast<uint4*>(sm + C::OFF_C + off) = vc;
          *reinterpret_cast<uint4*>(sm + C::OFF_BL + off) = lb;
          *reinterpret_cast<uint4*>(sm + C::OFF_CL + off) = lc;
        }
      }
      if (tb == TB - 1) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          s_carry[((ck + 1) & 1) * 64 + 4 * pg + q] = reduce_angle(base[q] + phl[TPT - 1][q]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(!ok)) break;

    // ------------------------------------------------------------ GEMM1: S = C~ B~^T
    // (C_hi + C_lo)(B_hi + B_lo)^T without the lo*lo term.
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const uint32_t ko = (ks >> 2) * 16384u + (ks & 3) * 32u;
        tc_mma_ss(tS, sdesc_sw128(sC + ko, 16, 1024), sdesc_sw128(sB + ko, 16, 1024), I_S, ks > 0);
        tc_mma_ss(tS, sdesc_sw128(sC + ko, 16, 1024), sdesc_sw128(sBl + ko, 16, 1024), I_S, 1);
        tc_mma_ss(tS, sdesc_sw128(sCl + ko, 16, 1024), sdesc_sw128(sB + ko, 16, 1024), I_S, 1);
      }
      tc_commit(bar_mma);
    }
    ok = mbar_wait(bar_mma, mma_count & 1) && ok;
    ++mma_count;
    tc_fence_after();

    // ------------------------------------------------------------ mask (registers)
    uint32_t pkh[32], pkl[32];  // this thread's 64 masked scores as bf16 (hi, lo) pairs
    {
      const int i = trow >> C::kLogR;
      const float ell_i = s_ell[i], gam_i = s_gam[i];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t sv[32];
        tmem_ld32(tS + lane_off + 64 * half + 32 * h2, sv);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float m2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int col = 64 * half + 32 * h2 + c + e;
            const int j = col >> C::kLogR;
            float m = 0.f;
            if (j < i) m = ex2(ell_i - s_ell[j]) * s_wgt[j];
            else if (j == i) m = gam_i;
            m2[e] = m * __uint_as_float(sv[c + e]);
          }
          split2(m2[0], m2[1], pkh[16 * h2 + c / 2], pkl[16 * h2 + c / 2]);
        }
      }
    }
    // Scale B~ rows by d_j (for GEMM4) and C~ rows by e^{l_i} (for GEMM3), in place:
    // recombine hi + lo in fp32, scale, split again.
    {
      const int row = tid & 127;
      const int i = row >> C::kLogR;
      const float fb = s_dsc[i], fc = s_eL[i];
      const int hh = tid >> 7;
#pragma unroll
      for (int cc = 0; cc < NB * 4; ++cc) {
        const int chunk = hh * NB * 4 + cc;  // 0 .. NB*8-1
        const uint32_t off = (chunk >> 3) * 16384u + sw128(row, chunk & 7);
        uint4 vb = *reinterpret_cast<const uint4*>(sm + C::OFF_B + off);
        uint4 vc = *reinterpret_cast<const uint4*>(sm + C::OFF_C + off);
        uint4 lb = *reinterpret_cast<const uint4*>(sm + C::OFF_BL + off);
        uint4 lc = *reinterpret_cast<const uint4*>(sm + C::OFF_CL + off);
        uint32_t* wb = reinterpret_cast<uint32_t*>(&vb);
        uint32_t* wc = reinterpret_cast<uint32_t*>(&vc);
        uint32_t* wlb = reinterpret_cast<uint32_t*>(&lb);
        uint32_t* wlc = reinterpret_cast<uint32_t*>(&lc);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 bh_ = unpack_bf16x2(wb[q]), bl_ = unpack_bf16x2(wlb[q]);
          const float2 ch_ = unpack_bf16x2(wc[q]), cl_ = unpack_bf16x2(wlc[q]);
          split2(fb * (bh_.x + bl_.x), fb * (bh_.y + bl_.y), wb[q], wlb[q]);
          split2(fc * (ch_.x + cl_.x), fc * (ch_.y + cl_.y), wc[q], wlc[q]);
        }
        *reinterpret_cast<uint4*>(sm + C::OFF_B + off) = vb;
        *reinterpret_cast<uint4*>(sm + C::OFF_C + off) = vc;
        *reinterpret_cast<uint4*>(sm + C::OFF_BL + off) = lb;
        *reinterpret_cast<uint4*>(sm + C::OFF_CL + off) = lc;
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(!ok)) break;

    // ------------------------------------------------------------ GEMM3 + GEMM4
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const uint32_t ka = (ks >> 2) * 16384u + (ks & 3) * 32u;
        const uint32_t kh = (ks >> 2) * 8192u + (ks & 3) * 32u;
        tc_mma_ss(tY, sdesc_sw128(sC + ka, 16, 1024), sdesc_sw128(sH + kh, 16, 1024), I_CH, ks > 0);
        tc_mma_ss(tY, sdesc_sw128(sC + ka, 16, 1024), sdesc_sw128(sHl + kh, 16, 1024), I_CH, 1);
        tc_mma_ss(tY, sdesc_sw128(sCl + ka, 16, 1024), sdesc_sw128(sH + kh, 16, 1024), I_CH, 1);
      }
#pragma unroll
      for (int ks = 0; ks < kRows / 16; ++ks) {
        const uint32_t kr = ks * 2048u;
        tc_mma_ss(tU, sdesc_sw128(sB + kr, 16384, 1024), sdesc_sw128(sX + kr, 16384, 1024), I_U,
                  ks > 0);
        tc_mma_ss(tU, sdesc_sw128(sBl + kr, 16384, 1024), sdesc_sw128(sX + kr, 16384, 1024), I_U, 1);
      }
      tc_commit(bar_mma);
    }
    ok = mbar_wait(bar_mma, mma_count & 1) && ok;
    ++mma_count;
    tc_fence_after();

    // P -> shared memory (K-major A operand of GEMM2, in B~'s hi and lo buffers)
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
      const uint32_t off = half * 16384u + sw128(trow, c8);
      *reinterpret_cast<uint4*>(sm + C::OFF_P + off) =
          make_uint4(pkh[4 * c8], pkh[4 * c8 + 1], pkh[4 * c8 + 2], pkh[4 * c8 + 3]);
      *reinterpret_cast<uint4*>(sm + C::OFF_PL + off) =
          make_uint4(pkl[4 * c8], pkl[4 * c8 + 1], pkl[4 * c8 + 2], pkl[4 * c8 + 3]);
    }
    // state: H <- e^{l_last} H + U
    if ((warp & 3) * 32 < NS) {
      const float eLast = s_scal[0];
      uint32_t hv[32], uv[32];
      tmem_ld32(tHc + lane_off + 32 * half, hv);
      tmem_ld32(tU + lane_off + 32 * half, uv);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j)
        hv[j] = __float_as_uint(fmaf(eLast, __uint_as_float(hv[j]), __uint_as_float(uv[j])));
      put_state(hv);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(!ok)) break;

    // ------------------------------------------------------------ GEMM2: Y += (P_hi + P_lo) X
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < kRows / 16; ++ks) {
        const uint32_t ka = (ks >> 2) * 16384u + (ks & 3) * 32u;
        const uint64_t bx = sdesc_sw128(sX + ks * 2048u, 16384, 1024);
        tc_mma_ss(tY, sdesc_sw128(sP + ka, 16, 1024), bx, I_PX, 1);
        tc_mma_ss(tY, sdesc_sw128(sPl + ka, 16, 1024), bx, I_PX, 1);
      }
      tc_commit(bar_mma);
    }
    ok = mbar_wait(bar_mma, mma_count & 1) && ok;
    ++mma_count;
    tc_fence_after();
    if (tid == 0 && ok && ck + 1 < nchunks) {
      fence_proxy_async_smem();
      issue_tma(ck + 1);
    }

    // ------------------------------------------------------------ y
    {
      uint32_t yv[32];
      tmem_ld32(tY + lane_off + 32 * half, yv);
      tmem_ld_wait();
      const int i = trow >> C::kLogR, r = trow & (R - 1);
      const int t = t0 + i;
      if (t < T) {
        const size_t o = (((static_cast<size_t>(b) * T + t) * H + head) * R + r) * kP + 32 * half;
        if (p.out_bf16) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.y) + o);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[q] = make_uint4(
                pack_bf16x2(__uint_as_float(yv[8 * q + 0]), __uint_as_float(yv[8 * q + 1])),
                pack_bf16x2(__uint_as_float(yv[8 * q + 2]), __uint_as_float(yv[8 * q + 3])),
                pack_bf16x2(__uint_as_float(yv[8 * q + 4]), __uint_as_float(yv[8 * q + 5])),
                pack_bf16x2(__uint_as_float(yv[8 * q + 6]), __uint_as_float(yv[8 * q + 7])));
        } else {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.y) + o);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(__uint_as_float(yv[4 * q]), __uint_as_float(yv[4 * q + 1]),
                                 __uint_as_float(yv[4 * q + 2]), __uint_as_float(yv[4 * q + 3]));
        }
      }
    }
    tc_fence_before();
    if (__syncthreads_or(!ok)) break;
  }

  if (!ok) {
    if (tid == 0) atomicOr(p.status, kDevTimeout);
  } else {
    // ------------------------------------------------------------ exit state
    if (p.hT && (warp & 3) * 32 < NS) {
      uint32_t hv[32];
      tmem_ld32(tHc + lane_off + 32 * half, hv);
      tmem_ld_wait();
      float4* dst =
          reinterpret_cast<float4*>(p.hT + (static_cast<size_t>(bh) * NS + trow) * kP + 32 * half);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        dst[q] = make_float4(__uint_as_float(hv[4 * q]), __uint_as_float(hv[4 * q + 1]),
                             __uint_as_float(hv[4 * q + 2]), __uint_as_float(hv[4 * q + 3]));
    }
    if (p.phiT)
      for (int k = tid; k < K; k += kThreads)
        p.phiT[static_cast<size_t>(bh) * K + k] = s_carry[(nchunks & 1) * 64 + k];
    if (p.prevBT)
      for (int e = tid; e < R * NS; e += kThreads)
        p.prevBT[static_cast<size_t>(bh) * R * NS + e] =
            T > 0 ? p.B[((static_cast<size_t>(b) * T + T - 1) * H + head) * R * NS + e]
                  : (p.prevB0 ? p.prevB0[static_cast<size_t>(bh) * R * NS + e] : __float2bfloat16_rn(0.f));
    if (p.prevxT)
      for (int e = tid; e < R * kP; e += kThreads)
        p.prevxT[static_cast<size_t>(bh) * R * kP + e] =
            T > 0 ? p.x[((static_cast<size_t>(b) * T + T - 1) * H + head) * R * kP + e]
                  : (p.prevx0 ? p.prevx0[static_cast<size_t>(bh) * R * kP + e] : __float2bfloat16_rn(0.f));
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
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
