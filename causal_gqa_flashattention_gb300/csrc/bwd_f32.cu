// bwd_f32.cu -- backward for fp32 inputs (d = 64) on tcgen05 kind::tf32.
//
// Same gradient as the bf16 path ("NanoEuler: Hand-writing GPT-2 in Pure
// C/CUDA", section "Hand-written Backpropagation"), laid out for the tf32
// tensor-core rule that both smem operands be K-major:
//  transpose_tf32   writes Q^T, dO^T [heads][d][N] and K^T [kv heads][d][N]
//                   into the workspace, rounded to tf32 (nearest);
//  dkdv_f32_kernel  one CTA per (batch, KV head, key tile j), walking the
//                   group's heads and query tiles i >= j:
//                     S^T = K Q^T, dP^T = V dO^T          (SS, K-major)
//                     P^T, dS^T written back over S^T, dP^T in TMEM (fp32)
//                     dV += P^T (dO^T)^T, dK += dS^T (Q^T)^T   (TS)
//  dq_f32_kernel    one CTA per (batch, head, query tile i), walking key
//                   tiles j <= i:  S = Q K^T, dP = dO V^T (SS), dS written
//                   over dP in TMEM, dQ += dS (K^T)^T (TS); dQ stored once.
// Each query tile's dQ is owned by one CTA, so this path needs no fp32
// accumulator and no reduction.
#include "nea_internal.h"
#include "ptx.cuh"
#include "rope.cuh"

namespace nea {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int D = 64;                     // head_dim of the fp32 path
constexpr int BLK = kTile * 128;          // [128 rows][128 B] block (16 KB)
constexpr int TILE = 2 * BLK;             // [128 rows][64 fp32]
constexpr int TBLK = D * 128;             // [64 rows][128 B] block of a transposed tile (8 KB)
constexpr int TTILE = 4 * TBLK;           // [64 rows][128 fp32]

// ---------------------------------------------------------------- transpose
// src [heads][N][64] -> dst [heads][64][npad], tf32-rounded, zeros in the
// columns n >= N (npad = N rounded up to whole 128-row tiles, so that every
// row of dst starts 16-byte aligned for TMA).  Block = 64 columns n of dst x
// all 64 rows, 256 threads.
__global__ void __launch_bounds__(256) transpose_tf32_kernel(const float* __restrict__ src,
                                                             float* __restrict__ dst, int N,
                                                             int npad) {
  __shared__ float tile[64][65];
  const int n0 = blockIdx.x * 64;
  const size_t head = blockIdx.y;
  const float* s = src + (head * N + n0) * D;
  for (int e = threadIdx.x; e < 64 * 64; e += 256) {
    const int r = e / 64, c = e % 64;
    tile[r][c] = n0 + r < N ? s[static_cast<size_t>(r) * D + c] : 0.f;
  }
  __syncthreads();
  float* d = dst + head * D * npad + n0;
  for (int e = threadIdx.x; e < 64 * 64; e += 256) {
    const int c = e / 64, r = e % 64;  // write row c of dst, 64 consecutive n
    d[static_cast<size_t>(c) * npad + r] = __uint_as_float(tf32_rna(tile[r][c]));
  }
}

// K-major descriptor of K-step k (8 tf32 = 32 B) in a tile made of blocks of
// `blk` bytes that each hold 32 K-elements of every row.
__device__ __forceinline__ uint64_t kmaj(uint32_t base, int k, int blk) {
  return sdesc_sw128(base + (k / 4) * blk + (k % 4) * 32, 16, 1024);
}

// ---------------------------------------------------------------- dK, dV
enum : int { F_KV = 0, F_QFULL, F_DOFULL, F_QEMPTY, F_SFULL, F_DPFULL, F_PFULL, F_DSFULL, F_FINAL,
             F_DRAIN, F_NBARS };

struct DkdvCfg {
  static constexpr int OFF_K = 0, OFF_V = TILE, OFF_Q = 2 * TILE, OFF_QT = 3 * TILE;
  static constexpr int OFF_DO = 3 * TILE + TTILE, OFF_DOT = 4 * TILE + TTILE;
  static constexpr int OFF_L2 = 4 * TILE + 2 * TTILE, OFF_DS = OFF_L2 + 512;
  static constexpr int SMEM_BYTES = 1024 + OFF_DS + 512;
  static constexpr int S_COL = 0, DP_COL = 128, DV_COL = 256, DK_COL = 320;
  static constexpr int THREADS = 384;
};

__global__ void __launch_bounds__(DkdvCfg::THREADS, 1)
    dkdv_f32_kernel(const __grid_constant__ BwdArgs a, const __grid_constant__ CUtensorMap tmQt,
                    const __grid_constant__ CUtensorMap tmdOt) {
  using C = DkdvCfg;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t bars[F_NBARS];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = (a.N + kTile - 1) / kTile, BG = a.B * a.Hkv, G = a.H / a.Hkv;
  const int j = blockIdx.x / BG, bg = blockIdx.x % BG;
  const int b = bg / a.Hkv, g = bg % a.Hkv;
  const int i0 = a.causal ? j : 0, nI = T - i0, nsteps = G * nI;
  const uint32_t base = smem_u32(smem);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  volatile int* abort = &abort_sh;
  unsigned int* status = a.status;
  auto step_hi = [&](int n, int& h, int& i) {
    h = g * G + n / nI;
    i = i0 + n % nI;
  };
  if (threadIdx.x == 0) {
    abort_sh = 0;
    for (int k = 0; k < F_NBARS; ++k) mbar_init(bar(k), 1);
    mbar_init(bar(F_QEMPTY), 1 + 8);
    mbar_init(bar(F_PFULL), 256);
    mbar_init(bar(F_DSFULL), 256);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    if (lane == 0) {
      const int kvh = b * a.Hkv + g;
      mbar_expect_tx(bar(F_KV), 2 * TILE);
      for (int k = 0; k < 2; ++k) {
        tma_load_3d(base + C::OFF_K + k * BLK, &a.tmK, bar(F_KV), 32 * k, j * kTile, kvh);
        tma_load_3d(base + C::OFF_V + k * BLK, &a.tmV, bar(F_KV), 32 * k, j * kTile, kvh);
      }
      int issued = 0;
      for (int n = 0; n < nsteps; ++n) {
        if (n > 0 && !mbar_wait(bar(F_QEMPTY), (n - 1) & 1, abort, 40, status)) break;
        int h, i;
        step_hi(n, h, i);
        const int bh = b * a.H + h;
        const size_t row0 = (static_cast<size_t>(bh) * T + i) * kTile;  // padded per-row terms
        mbar_expect_tx(bar(F_QFULL), TILE + TTILE + 512);
        for (int k = 0; k < 2; ++k)
          tma_load_3d(base + C::OFF_Q + k * BLK, &a.tmQ, bar(F_QFULL), 32 * k, i * kTile, bh);
        for (int k = 0; k < 4; ++k)
          tma_load_3d(base + C::OFF_QT + k * TBLK, &tmQt, bar(F_QFULL), i * kTile + 32 * k, 0, bh);
        bulk_load(base + C::OFF_L2, a.lse2 + row0, 512, bar(F_QFULL));
        mbar_expect_tx(bar(F_DOFULL), TILE + TTILE + 512);
        for (int k = 0; k < 2; ++k)
          tma_load_3d(base + C::OFF_DO + k * BLK, &a.tmdO, bar(F_DOFULL), 32 * k, i * kTile, bh);
        for (int k = 0; k < 4; ++k)
          tma_load_3d(base + C::OFF_DOT + k * TBLK, &tmdOt, bar(F_DOFULL), i * kTile + 32 * k, 0,
                      bh);
        bulk_load(base + C::OFF_DS, a.delta + row0, 512, bar(F_DOFULL));
        issued = n + 1;
      }
      mbar_wait_drain(bar(F_KV), 0, 41, status);
      if (issued > 0) {
        mbar_wait_drain(bar(F_QFULL), (issued - 1) & 1, 41, status);
        mbar_wait_drain(bar(F_DOFULL), (issued - 1) & 1, 41, status);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idS = make_idesc<MmaKind::kTF32>(128, 128, false, false);
      constexpr uint32_t idG = make_idesc<MmaKind::kTF32>(128, D, false, false);
      bool ok = mbar_wait(bar(F_KV), 0, abort, 42, status);
      for (int n = 0; ok && n < nsteps; ++n) {
        const uint32_t ph = n & 1;
        if (!mbar_wait(bar(F_QFULL), ph, abort, 43, status)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ss<MmaKind::kTF32>(tmem + C::S_COL, kmaj(base + C::OFF_K, k, BLK),
                                 kmaj(base + C::OFF_Q, k, BLK), idS, k > 0 ? 1u : 0u);
        mma_commit(bar(F_SFULL));
        if (!mbar_wait(bar(F_DOFULL), ph, abort, 44, status)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ss<MmaKind::kTF32>(tmem + C::DP_COL, kmaj(base + C::OFF_V, k, BLK),
                                 kmaj(base + C::OFF_DO, k, BLK), idS, k > 0 ? 1u : 0u);
        mma_commit(bar(F_DPFULL));
        if (!mbar_wait(bar(F_PFULL), ph, abort, 45, status)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 16; ++k)  // dV += P^T dO, K = 128 queries
          mma_ts<MmaKind::kTF32>(tmem + C::DV_COL, tmem + C::S_COL + k * 8,
                                 kmaj(base + C::OFF_DOT, k, TBLK), idG, (n > 0 || k > 0) ? 1u : 0u);
        if (!mbar_wait(bar(F_DSFULL), ph, abort, 46, status)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 16; ++k)  // dK += dS^T Q
          mma_ts<MmaKind::kTF32>(tmem + C::DK_COL, tmem + C::DP_COL + k * 8,
                                 kmaj(base + C::OFF_QT, k, TBLK), idG, (n > 0 || k > 0) ? 1u : 0u);
        mma_commit(bar(F_QEMPTY));
      }
      mma_commit(bar(F_FINAL));
      mma_commit(bar(F_DRAIN));
      mbar_wait_drain(bar(F_DRAIN), 0, 47, status);
    }
  } else if (warp >= 4) {
    const int half = (warp - 4) >> 2, quad = warp & 3;
    const int kr = quad * 32 + lane, q0 = 64 * half;
    const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const float c = a.scale * kLog2e;
    const float* l2s = reinterpret_cast<const float*>(smem + C::OFF_L2) + q0;
    const float* dss = reinterpret_cast<const float*>(smem + C::OFF_DS) + q0;
    bool ok = true;
    for (int n = 0; n < nsteps; ++n) {
      const uint32_t ph = n & 1;
      int h, i;
      step_hi(n, h, i);
      if (!mbar_wait_warp(bar(F_QFULL), ph, abort, 48, status) ||
          !mbar_wait_warp(bar(F_SFULL), ph, abort, 49, status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t u0[32], u1[32];
      tmem_ld32(trow + C::S_COL + q0, u0);
      tmem_ld32(trow + C::S_COL + q0 + 32, u1);
      tmem_ld_wait(u0);
      reg_fence(u1);
      const bool diag = a.causal && i == j;
      const bool kdead = !a.causal && j * kTile + kr >= a.N;  // key past N, no causal mask
      float p[64];
#pragma unroll
      for (int t = 0; t < 64; ++t) {
        const float sv = __uint_as_float(t < 32 ? u0[t] : u1[t - 32]);
        float pv = ex2(fmaf(sv, c, l2s[t]));
        if ((diag && q0 + t < kr) || kdead) pv = 0.f;
        p[t] = pv;
      }
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        u0[t] = tf32_rna(p[t]);
        u1[t] = tf32_rna(p[32 + t]);
      }
      tmem_st32(trow + C::S_COL + q0, u0);
      tmem_st32(trow + C::S_COL + q0 + 32, u1);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(F_PFULL));
      if (!mbar_wait_warp(bar(F_DOFULL), ph, abort, 50, status) ||
          !mbar_wait_warp(bar(F_DPFULL), ph, abort, 51, status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_ld32(trow + C::DP_COL + q0, u0);
      tmem_ld32(trow + C::DP_COL + q0 + 32, u1);
      tmem_ld_wait(u0);
      reg_fence(u1);
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        u0[t] = tf32_rna(p[t] * fmaf(__uint_as_float(u0[t]), a.scale, -dss[t]));
        u1[t] = tf32_rna(p[32 + t] * fmaf(__uint_as_float(u1[t]), a.scale, -dss[32 + t]));
      }
      tmem_st32(trow + C::DP_COL + q0, u0);
      tmem_st32(trow + C::DP_COL + q0 + 32, u1);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(F_DSFULL));
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(F_QEMPTY));
    }
    if (ok) ok = mbar_wait_warp(bar(F_FINAL), 0, abort, 52, status);
    if (ok) {
      tc_fence_after();
      const bool row_ok = j * kTile + kr < a.N;
      const size_t row =
          (static_cast<size_t>(b) * a.Hkv + g) * a.N + static_cast<size_t>(j) * kTile + kr;
      float* dst = static_cast<float*>(half == 0 ? a.dV : a.dK) + row * D;
      const uint32_t col = half == 0 ? C::DV_COL : C::DK_COL;
      // dK of rotated keys -> dK of the caller's keys (RoPE)
      const float2* rcs = (half == 1 && row_ok && a.rope_cs != nullptr)
                              ? a.rope_cs + static_cast<size_t>(j * kTile + kr) * (D / 2)
                              : nullptr;
#pragma unroll
      for (int cc = 0; cc < D; cc += 32) {
        uint32_t v[32];
        tmem_ld32(trow + col + cc, v);
        tmem_ld_wait(v);
        if (rcs != nullptr) {
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            float x0 = __uint_as_float(v[2 * t]), x1 = __uint_as_float(v[2 * t + 1]);
            rope_inv(x0, x1, __ldg(rcs + cc / 2 + t));
            v[2 * t] = __float_as_uint(x0);
            v[2 * t + 1] = __float_as_uint(x1);
          }
        }
#pragma unroll
        for (int t4 = 0; t4 < 8; ++t4)
          if (row_ok)
            *reinterpret_cast<uint4*>(dst + cc + 4 * t4) =
                make_uint4(v[4 * t4], v[4 * t4 + 1], v[4 * t4 + 2], v[4 * t4 + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- dQ
enum : int { Q_QFULL = 0, Q_KTFULL, Q_KTEMPTY, Q_SFULL, Q_DPFULL, Q_DSFULL, Q_FINAL, Q_DRAIN,
             Q_KFULL, Q_NBARS = Q_KFULL + 6 };  // KFULL[2], VFULL[2], KVEMPTY[2]

struct DqCfg {
  static constexpr int OFF_Q = 0, OFF_DO = TILE, OFF_KV = 2 * TILE;  // stage s: K, V
  static constexpr int OFF_KT = 6 * TILE;
  static constexpr int SMEM_BYTES = 1024 + OFF_KT + TTILE;
  static constexpr int S_COL = 0, DP_COL = 128, DQ_COL = 256;
  static constexpr int THREADS = 384;
};

__global__ void __launch_bounds__(DqCfg::THREADS, 1)
    dq_f32_kernel(const __grid_constant__ BwdArgs a, const __grid_constant__ CUtensorMap tmKt) {
  using C = DqCfg;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t bars[Q_NBARS];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = (a.N + kTile - 1) / kTile, BH = a.B * a.H;
  const int it = a.causal ? (T - 1 - blockIdx.x / BH) : (blockIdx.x / BH);  // longest first
  const int bh = blockIdx.x % BH;
  const int b = bh / a.H, h = bh % a.H;
  const int kvh = b * a.Hkv + h / (a.H / a.Hkv);
  const int nkv = a.causal ? it + 1 : T;
  const uint32_t base = smem_u32(smem);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  auto kfull = [&](int s) { return bar(Q_KFULL + s); };
  auto vfull = [&](int s) { return bar(Q_KFULL + 2 + s); };
  auto kvempty = [&](int s) { return bar(Q_KFULL + 4 + s); };
  auto sK = [&](int s) { return base + C::OFF_KV + 2 * s * TILE; };
  auto sV = [&](int s) { return base + C::OFF_KV + (2 * s + 1) * TILE; };
  volatile int* abort = &abort_sh;
  unsigned int* status = a.status;
  if (threadIdx.x == 0) {
    abort_sh = 0;
    for (int k = 0; k < Q_NBARS; ++k) mbar_init(bar(k), 1);
    mbar_init(bar(Q_DSFULL), 256);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    if (lane == 0) {
      mbar_expect_tx(bar(Q_QFULL), 2 * TILE);
      for (int k = 0; k < 2; ++k) {
        tma_load_3d(base + C::OFF_Q + k * BLK, &a.tmQ, bar(Q_QFULL), 32 * k, it * kTile, bh);
        tma_load_3d(base + C::OFF_DO + k * BLK, &a.tmdO, bar(Q_QFULL), 32 * k, it * kTile, bh);
      }
      int issued = 0, kt_issued = 0;
      for (int jj = 0; jj < nkv; ++jj) {
        const int s = jj & 1;
        if (jj >= 2 && !mbar_wait(kvempty(s), ((jj >> 1) - 1) & 1, abort, 60, status)) break;
        mbar_expect_tx(kfull(s), TILE);
        for (int k = 0; k < 2; ++k)
          tma_load_3d(sK(s) + k * BLK, &a.tmK, kfull(s), 32 * k, jj * kTile, kvh);
        mbar_expect_tx(vfull(s), TILE);
        for (int k = 0; k < 2; ++k)
          tma_load_3d(sV(s) + k * BLK, &a.tmV, vfull(s), 32 * k, jj * kTile, kvh);
        issued = jj + 1;
        if (jj >= 1 && !mbar_wait(bar(Q_KTEMPTY), (jj - 1) & 1, abort, 61, status)) break;
        mbar_expect_tx(bar(Q_KTFULL), TTILE);
        for (int k = 0; k < 4; ++k)
          tma_load_3d(base + C::OFF_KT + k * TBLK, &tmKt, bar(Q_KTFULL), jj * kTile + 32 * k, 0,
                      kvh);
        kt_issued = jj + 1;
      }
      mbar_wait_drain(bar(Q_QFULL), 0, 62, status);
      for (int jj = issued - 2 > 0 ? issued - 2 : 0; jj < issued; ++jj) {
        mbar_wait_drain(kfull(jj & 1), (jj >> 1) & 1, 62, status);
        mbar_wait_drain(vfull(jj & 1), (jj >> 1) & 1, 62, status);
      }
      if (kt_issued > 0) mbar_wait_drain(bar(Q_KTFULL), (kt_issued - 1) & 1, 62, status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idS = make_idesc<MmaKind::kTF32>(128, 128, false, false);
      constexpr uint32_t idG = make_idesc<MmaKind::kTF32>(128, D, false, false);
      bool ok = mbar_wait(bar(Q_QFULL), 0, abort, 63, status);
      for (int jj = 0; ok && jj < nkv; ++jj) {
        const int s = jj & 1;
        const uint32_t ph = (jj >> 1) & 1;
        if (!mbar_wait(kfull(s), ph, abort, 64, status)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ss<MmaKind::kTF32>(tmem + C::S_COL, kmaj(base + C::OFF_Q, k, BLK), kmaj(sK(s), k, BLK),
                                 idS, k > 0 ? 1u : 0u);
        mma_commit(bar(Q_SFULL));
        if (!mbar_wait(vfull(s), ph, abort, 65, status)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ss<MmaKind::kTF32>(tmem + C::DP_COL, kmaj(base + C::OFF_DO, k, BLK),
                                 kmaj(sV(s), k, BLK), idS, k > 0 ? 1u : 0u);
        mma_commit(bar(Q_DPFULL));
        mma_commit(kvempty(s));
        if (!mbar_wait(bar(Q_DSFULL), jj & 1, abort, 66, status)) break;
        if (!mbar_wait(bar(Q_KTFULL), jj & 1, abort, 67, status)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 16; ++k)  // dQ += dS K, K = 128 keys
          mma_ts<MmaKind::kTF32>(tmem + C::DQ_COL, tmem + C::DP_COL + k * 8,
                                 kmaj(base + C::OFF_KT, k, TBLK), idG, (jj > 0 || k > 0) ? 1u : 0u);
        mma_commit(bar(Q_KTEMPTY));
      }
      mma_commit(bar(Q_FINAL));
      mma_commit(bar(Q_DRAIN));
      mbar_wait_drain(bar(Q_DRAIN), 0, 68, status);
    }
  } else if (warp >= 4) {
    const int half = (warp - 4) >> 2, quad = warp & 3;
    const int r = quad * 32 + lane, k0 = 64 * half;  // query row, first key column
    const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const float c = a.scale * kLog2e;
    const size_t row = static_cast<size_t>(bh) * a.N + static_cast<size_t>(it) * kTile + r;
    const size_t prow = (static_cast<size_t>(bh) * T + it) * kTile + r;  // padded per-row terms
    const float nl2 = a.lse2[prow], dsr = a.delta[prow];
    const bool row_ok = it * kTile + r < a.N;
    bool ok = true;
    for (int jj = 0; jj < nkv; ++jj) {
      if (!mbar_wait_warp(bar(Q_SFULL), jj & 1, abort, 69, status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t u0[32], u1[32];
      tmem_ld32(trow + C::S_COL + k0, u0);
      tmem_ld32(trow + C::S_COL + k0 + 32, u1);
      tmem_ld_wait(u0);
      reg_fence(u1);
      const bool diag = a.causal && jj == it;
      // keys past N: masked with the diagonal under the causal mask, here otherwise
      const int klim = (!a.causal && jj == T - 1) ? a.N - 1 - jj * kTile : kTile;
      float p[64];
#pragma unroll
      for (int t = 0; t < 64; ++t) {
        const float sv = __uint_as_float(t < 32 ? u0[t] : u1[t - 32]);
        float pv = ex2(fmaf(sv, c, nl2));
        if ((diag && k0 + t > r) || k0 + t > klim) pv = 0.f;
        p[t] = pv;
      }
      if (!mbar_wait_warp(bar(Q_DPFULL), jj & 1, abort, 70, status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_ld32(trow + C::DP_COL + k0, u0);
      tmem_ld32(trow + C::DP_COL + k0 + 32, u1);
      tmem_ld_wait(u0);
      reg_fence(u1);
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        u0[t] = tf32_rna(p[t] * fmaf(__uint_as_float(u0[t]), a.scale, -dsr));
        u1[t] = tf32_rna(p[32 + t] * fmaf(__uint_as_float(u1[t]), a.scale, -dsr));
      }
      tmem_st32(trow + C::DP_COL + k0, u0);
      tmem_st32(trow + C::DP_COL + k0 + 32, u1);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(Q_DSFULL));
    }
    if (ok) ok = mbar_wait_warp(bar(Q_FINAL), 0, abort, 71, status);
    if (ok) {
      tc_fence_after();
      float* dst = static_cast<float*>(a.dQ) + row * D + 32 * half;
      uint32_t v[32];
      tmem_ld32(trow + C::DQ_COL + 32 * half, v);
      tmem_ld_wait(v);
      if (row_ok && a.rope_cs != nullptr) {  // dQ of rotated queries -> caller's queries
        const float2* rcs = a.rope_cs + static_cast<size_t>(it * kTile + r) * (D / 2) + 16 * half;
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          float x0 = __uint_as_float(v[2 * t]), x1 = __uint_as_float(v[2 * t + 1]);
          rope_inv(x0, x1, __ldg(rcs + t));
          v[2 * t] = __float_as_uint(x0);
          v[2 * t + 1] = __float_as_uint(x1);
        }
      }
#pragma unroll
      for (int t4 = 0; t4 < 8; ++t4)
        if (row_ok)
          *reinterpret_cast<uint4*>(dst + 4 * t4) =
              make_uint4(v[4 * t4], v[4 * t4 + 1], v[4 * t4 + 2], v[4 * t4 + 3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_transpose_f32(const float* src, float* dst, long long heads, int N,
                                 cudaStream_t stream) {
  const int npad = (N + kTile - 1) / kTile * kTile;
  transpose_tf32_kernel<<<dim3(npad / 64, static_cast<unsigned>(heads)), 256, 0, stream>>>(
      src, dst, N, npad);
  return cudaGetLastError();
}

cudaError_t launch_bwd_main_f32(const BwdArgs& a, const CUtensorMap& tmQt,
                                const CUtensorMap& tmdOt, const CUtensorMap& tmKt,
                                cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(dkdv_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       DkdvCfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(dq_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           DqCfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const unsigned T = static_cast<unsigned>((a.N + kTile - 1) / kTile);
  dkdv_f32_kernel<<<static_cast<unsigned>(a.B) * a.Hkv * T, DkdvCfg::THREADS, DkdvCfg::SMEM_BYTES,
                    stream>>>(a, tmQt, tmdOt);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dq_f32_kernel<<<static_cast<unsigned>(a.B) * a.H * T, DqCfg::THREADS, DqCfg::SMEM_BYTES,
                  stream>>>(a, tmKt);
  return cudaGetLastError();
}

}  // namespace nea
