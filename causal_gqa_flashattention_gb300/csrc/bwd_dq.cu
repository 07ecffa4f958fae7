// bwd_dq.cu -- deterministic dQ for bf16 inputs.
//
// Same gradient as the main backward ("NanoEuler: Hand-writing GPT-2 in Pure
// C/CUDA", section "Hand-written Backpropagation"), with dQ owned by one CTA
// per (batch, head, 128-row query tile i): it walks the key tiles j in a fixed
// order, recomputes S = Q K_j^T and dP = dO V_j^T on the tensor cores, forms
// dS and accumulates dQ += dS K_j in tensor memory.  No partial sums cross
// CTAs, so dQ has the same bits on every run.  The main kernel runs in its
// dK / dV-only form beside it.  Costs two extra GEMMs (S, dP) per tile pair.
//
// Roles (384 threads): warp 0 TMA producer (Q, dO once; K_j / V_j in a
// two-stage ring), warp 1 MMA issuer and TMEM owner, warps 4..11 compute
// (two warpgroups over key halves; thread = query row, so the row's LSE and
// D terms are scalars).  TMEM: S [0,128), dP [128,256), dQ [256,256+d),
// dS (bf16 pairs, the A operand of dQ += dS K_j) [384,448).
#include <cuda_bf16.h>

#include "nea_internal.h"
#include "ptx.cuh"
#include "rope.cuh"

namespace nea {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

enum : int { D_QFULL = 0, D_SFULL, D_DPFULL, D_DSFULL, D_FINAL, D_DRAIN, D_KFULL,
             D_NBARS = D_KFULL + 6 };  // KFULL[2], VFULL[2], KVEMPTY[2]

template <int D>
struct DqCfg {
  static constexpr int NBLK = D / 64;
  static constexpr int BLK_BYTES = kTile * 128;  // [128 rows][128 B]
  static constexpr int TILE = NBLK * BLK_BYTES;  // [128 rows][D bf16]
  static constexpr int OFF_Q = 0, OFF_DO = TILE, OFF_KV = 2 * TILE;  // stage s: K, then V
  static constexpr int SMEM_BYTES = 1024 + OFF_KV + 4 * TILE;
  static constexpr int S_COL = 0, DP_COL = 128, DQ_COL = 256, DS_COL = 384;
  static constexpr int NK_QK = D / 16;  // K-steps over d
  static constexpr int THREADS = 384;
};

template <int D>
__global__ void __launch_bounds__(DqCfg<D>::THREADS, 1) dq_bf16_kernel(const __grid_constant__ BwdArgs a) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t bars[D_NBARS];
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
  auto kfull = [&](int s) { return bar(D_KFULL + s); };
  auto vfull = [&](int s) { return bar(D_KFULL + 2 + s); };
  auto kvempty = [&](int s) { return bar(D_KFULL + 4 + s); };
  auto sK = [&](int s) { return base + C::OFF_KV + 2 * s * C::TILE; };
  auto sV = [&](int s) { return base + C::OFF_KV + (2 * s + 1) * C::TILE; };
  volatile int* abort = &abort_sh;
  unsigned int* status = a.status;
  if (threadIdx.x == 0) {
    abort_sh = 0;
    for (int k = 0; k < D_NBARS; ++k) mbar_init(bar(k), 1);
    mbar_init(bar(D_DSFULL), 256);
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
      mbar_expect_tx(bar(D_QFULL), 2 * C::TILE);
      for (int k = 0; k < C::NBLK; ++k) {
        tma_load_3d(base + C::OFF_Q + k * C::BLK_BYTES, &a.tmQ, bar(D_QFULL), 64 * k, it * kTile, bh);
        tma_load_3d(base + C::OFF_DO + k * C::BLK_BYTES, &a.tmdO, bar(D_QFULL), 64 * k, it * kTile,
                    bh);
      }
      int issued = 0;
      for (int jj = 0; jj < nkv; ++jj) {
        const int s = jj & 1;
        if (jj >= 2 && !mbar_wait(kvempty(s), ((jj >> 1) - 1) & 1, abort, 80, status)) break;
        mbar_expect_tx(kfull(s), C::TILE);
        for (int k = 0; k < C::NBLK; ++k)
          tma_load_3d(sK(s) + k * C::BLK_BYTES, &a.tmK, kfull(s), 64 * k, jj * kTile, kvh);
        mbar_expect_tx(vfull(s), C::TILE);
        for (int k = 0; k < C::NBLK; ++k)
          tma_load_3d(sV(s) + k * C::BLK_BYTES, &a.tmV, vfull(s), 64 * k, jj * kTile, kvh);
        issued = jj + 1;
      }
      mbar_wait_drain(bar(D_QFULL), 0, 81, status);
      for (int jj = issued - 2 > 0 ? issued - 2 : 0; jj < issued; ++jj) {
        mbar_wait_drain(kfull(jj & 1), (jj >> 1) & 1, 81, status);
        mbar_wait_drain(vfull(jj & 1), (jj >> 1) & 1, 81, status);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idS = make_idesc<MmaKind::kBF16>(128, 128, false, false);
      constexpr uint32_t idQ = make_idesc<MmaKind::kBF16>(128, D, false, true);
      bool ok = mbar_wait(bar(D_QFULL), 0, abort, 82, status);
      for (int jj = 0; ok && jj < nkv; ++jj) {
        const int s = jj & 1;
        const uint32_t ph = (jj >> 1) & 1;
        // S = Q K_j^T (the compute warps read S_{jj-1} before DSFULL_{jj-1})
        if (!mbar_wait(kfull(s), ph, abort, 83, status)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < C::NK_QK; ++k) {
          const uint32_t off = (k / 4) * C::BLK_BYTES + (k % 4) * 32;
          mma_ss<MmaKind::kBF16>(tmem + C::S_COL, sdesc_sw128(base + C::OFF_Q + off, 16, 1024),
                                 sdesc_sw128(sK(s) + off, 16, 1024), idS, k > 0 ? 1u : 0u);
        }
        mma_commit(bar(D_SFULL));
        // dP = dO V_j^T
        if (!mbar_wait(vfull(s), ph, abort, 84, status)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < C::NK_QK; ++k) {
          const uint32_t off = (k / 4) * C::BLK_BYTES + (k % 4) * 32;
          mma_ss<MmaKind::kBF16>(tmem + C::DP_COL, sdesc_sw128(base + C::OFF_DO + off, 16, 1024),
                                 sdesc_sw128(sV(s) + off, 16, 1024), idS, k > 0 ? 1u : 0u);
        }
        mma_commit(bar(D_DPFULL));
        // dQ += dS K_j: A = dS (bf16 pairs in TMEM), B = K_j read N-major
        if (!mbar_wait(bar(D_DSFULL), jj & 1, abort, 85, status)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k)
          mma_ts<MmaKind::kBF16>(tmem + C::DQ_COL, tmem + C::DS_COL + k * 8,
                                 sdesc_sw128(sK(s) + k * 16 * 128, C::BLK_BYTES, 1024), idQ,
                                 (jj > 0 || k > 0) ? 1u : 0u);
        mma_commit(kvempty(s));
      }
      mma_commit(bar(D_FINAL));
      mma_commit(bar(D_DRAIN));
      mbar_wait_drain(bar(D_DRAIN), 0, 86, status);
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
      if (!mbar_wait_warp(bar(D_SFULL), jj & 1, abort, 87, status)) {
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
      if (!mbar_wait_warp(bar(D_DPFULL), jj & 1, abort, 88, status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_ld32(trow + C::DP_COL + k0, u0);
      tmem_ld32(trow + C::DP_COL + k0 + 32, u1);
      tmem_ld_wait(u0);
      reg_fence(u1);
      uint32_t pk[32];  // dS row, bf16 pairs (key 2t in the low half)
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const uint32_t x0 = t < 16 ? u0[2 * t] : u1[2 * t - 32];
        const uint32_t x1 = t < 16 ? u0[2 * t + 1] : u1[2 * t + 1 - 32];
        const float d0 = p[2 * t] * fmaf(__uint_as_float(x0), a.scale, -dsr);
        const float d1 = p[2 * t + 1] * fmaf(__uint_as_float(x1), a.scale, -dsr);
        pk[t] = pack_bf16(d0, d1);
      }
      // dS_{jj-1} was read by dQ_{jj-1}: that MMA precedes S_jj (SFULL_jj)
      tmem_st32(trow + C::DS_COL + 32 * half, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(D_DSFULL));
    }
    if (ok) ok = mbar_wait_warp(bar(D_FINAL), 0, abort, 89, status);
    if (ok) {
      tc_fence_after();
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dQ) + row * D + half * (D / 2);
      const float2* rcs = (row_ok && a.rope_cs != nullptr)
                              ? a.rope_cs + static_cast<size_t>(it * kTile + r) * (D / 2) +
                                    half * (D / 4)
                              : nullptr;
#pragma unroll
      for (int cc = 0; cc < D / 2; cc += 32) {
        uint32_t v[32];
        tmem_ld32(trow + C::DQ_COL + half * (D / 2) + cc, v);
        tmem_ld_wait(v);
        if (rcs != nullptr) {  // dQ of rotated queries -> the caller's queries
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            float x0 = __uint_as_float(v[2 * t]), x1 = __uint_as_float(v[2 * t + 1]);
            rope_inv(x0, x1, __ldg(rcs + cc / 2 + t));
            v[2 * t] = __float_as_uint(x0);
            v[2 * t + 1] = __float_as_uint(x1);
          }
        }
#pragma unroll
        for (int t4 = 0; t4 < 4; ++t4) {
          uint4 w;
          w.x = pack_bf16(__uint_as_float(v[8 * t4 + 0]), __uint_as_float(v[8 * t4 + 1]));
          w.y = pack_bf16(__uint_as_float(v[8 * t4 + 2]), __uint_as_float(v[8 * t4 + 3]));
          w.z = pack_bf16(__uint_as_float(v[8 * t4 + 4]), __uint_as_float(v[8 * t4 + 5]));
          w.w = pack_bf16(__uint_as_float(v[8 * t4 + 6]), __uint_as_float(v[8 * t4 + 7]));
          if (row_ok) *reinterpret_cast<uint4*>(dst + cc + 8 * t4) = w;
        }
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

template <int D>
cudaError_t launch_t(const BwdArgs& a, cudaStream_t stream) {
  using C = DqCfg<D>;
  auto kern = dq_bf16_kernel<D>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(a.B) * a.H * ((a.N + kTile - 1) / kTile);
  kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t stream) {
  if (a.dtype == 0 && a.d == 64) return launch_t<64>(a, stream);
  if (a.dtype == 0 && a.d == 128) return launch_t<128>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace nea
