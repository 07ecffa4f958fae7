// bwd.cu -- causal grouped-query FlashAttention backward on tcgen05 / TMEM.
//
// "NanoEuler: Hand-writing GPT-2 in Pure C/CUDA", section "Hand-written
// Backpropagation": every gradient is derived and written by hand.  For
// softmax attention with upstream dO:
//   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),  D = rowsum(dO o O),
//   dQ = scale dS K,  dK = scale dS^T Q,  P recomputed from the saved LSE.
//
// Three kernels:
//  bwd_pre   (HBM-bound)  Ds = scale * rowsum(dO o O), L2 = LSE * log2(e),
//                         and zeroes the fp32 dQ accumulator;
//  bwd_main  one CTA per (batch, KV head, 128-row key tile j); it walks the
//            group's query heads and the query tiles i >= j (causal):
//              warp 0      TMA producer (K_j, V_j once; Q_i, dO_i, L2_i, Ds_i
//                          per step into a ring)
//              warp 1      MMA issuer A (S^T, dP^T, dV) + TMEM owner
//              warp 2      MMA issuer B (dK, dQ)
//              warps 4..11 "compute", two warpgroups splitting the 128 query
//                          columns: thread = key row; P^T = exp2(S^T c - L2)
//                          to TMEM (bf16), dS^T = P^T o (scale dP^T - Ds) to
//                          smem (bf16, 128-B swizzle)
//              warps 12..15 "dQ": thread = query row; dQ_i partial TMEM ->
//                          smem -> TMA reduce-add (fp32) into the accumulator
//            MMAs per step: S^T = K Q^T, dP^T = V dO^T (both SS, K-major),
//            dV += P^T dO (TS), dK += dS^T Q (SS, B MN-major),
//            dQ = dS K (SS, A and B MN-major; same smem bytes as dS^T).
//            dK and dV stay in TMEM for the whole CTA: the sum over the
//            group's query heads needs no atomics.
//  bwd_post  dQ = bf16(dQ accumulator).
#include "nea_internal.h"
#include "ptx.cuh"
#include "rope.cuh"

namespace nea {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- preprocess
// Walks the per-head rows padded to whole 128-row tiles (npad = T * 128):
// padded row p = bh * npad + n.  Real rows (n < N) get Ds = scale * dO.O and
// L2 = LSE * log2(e); padding rows get Ds = 0 and L2 = +inf, so that the main
// kernel's exp2(S c - L2) is exactly 0 for them.  TPR threads per row, each
// owning 16 bytes of O and dO; every thread handles kPreRows rows with all
// loads (the row's LSE included) issued before any use, so that a wave of
// blocks waits for memory once.
constexpr int kPreRows = 4;
constexpr int kPreThreads = 256;

template <typename T, int D>
__global__ void __launch_bounds__(kPreThreads) bwd_pre_kernel(const T* __restrict__ O,
                                                      const T* __restrict__ dO,
                                                      const float* __restrict__ lse,
                                                      float* __restrict__ ds_row,
                                                      float* __restrict__ l2_row,
                                                      float* __restrict__ dq_acc, long long prows,
                                                      int N, int npad, float scale) {
  constexpr int EPV = 16 / sizeof(T);  // elements per 16-B vector
  constexpr int TPR = D / EPV;         // threads per row
  constexpr int RPB = kPreThreads / TPR;  // rows per block per pass
  static_assert(kTile % (RPB * kPreRows) == 0, "a block's rows must divide a tile");
  const int sub = threadIdx.x % TPR;
  // A block's RPB * kPreRows rows divide npad (a multiple of 128), so the
  // block lies inside one head: bh and the row offset are block-uniform.
  const long long pb = static_cast<long long>(blockIdx.x) * RPB * kPreRows;
  const long long bh = pb / npad;
  const int nb = static_cast<int>(pb - bh * npad) + threadIdx.x / TPR;
  const long long p0 = pb + threadIdx.x / TPR;
  uint4 ov[kPreRows], gv[kPreRows];
  float lv[kPreRows];
  long long rrow[kPreRows];  // unpadded row index, or -1 for padding / past the end
#pragma unroll
  for (int u = 0; u < kPreRows; ++u) {
    const long long p = p0 + static_cast<long long>(u) * RPB;
    const int n = nb + u * RPB;
    rrow[u] = (p < prows && n < N) ? bh * N + n : -1;
    lv[u] = 0.f;
    if (rrow[u] >= 0) {
      const size_t base = static_cast<size_t>(rrow[u]) * D + sub * EPV;
      ov[u] = __ldg(reinterpret_cast<const uint4*>(O + base));
      gv[u] = __ldg(reinterpret_cast<const uint4*>(dO + base));
      if (sub == 0) lv[u] = __ldg(lse + rrow[u]);
    } else {
      ov[u] = gv[u] = make_uint4(0, 0, 0, 0);
    }
  }
#pragma unroll
  for (int u = 0; u < kPreRows; ++u) {
    const long long p = p0 + static_cast<long long>(u) * RPB;
    float acc = 0.f;
    if constexpr (sizeof(T) == 2) {
      const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov[u]);
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv[u]);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 x = __bfloat1622float2(o2[k]), y = __bfloat1622float2(g2[k]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
    } else {
      const float* o4 = reinterpret_cast<const float*>(&ov[u]);
      const float* g4 = reinterpret_cast<const float*>(&gv[u]);
#pragma unroll
      for (int k = 0; k < 4; ++k) acc = fmaf(o4[k], g4[k], acc);
    }
    // every lane of the warp runs the shuffle (padding rows add zeros)
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (p < prows && sub == 0) {
      ds_row[p] = rrow[u] >= 0 ? acc * scale : 0.f;
      l2_row[p] = rrow[u] >= 0 ? lv[u] * kLog2e : INFINITY;
    }
    // zero this thread's share of the fp32 accumulator row (D floats)
    if (dq_acc != nullptr && rrow[u] >= 0) {
      float4* z = reinterpret_cast<float4*>(dq_acc + static_cast<size_t>(rrow[u]) * D);
#pragma unroll
      for (int k = sub; k < D / 4; k += TPR) z[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// ---------------------------------------------------------------- dQ cast
// Each thread converts kPostVecs groups of 8 fp32 -> 8 bf16.  With a RoPE
// table, the 4 pairs of a group are first turned back by their row's angles.
constexpr int kPostVecs = 4;
constexpr int kPostThreads = 256;

__global__ void __launch_bounds__(kPostThreads) bwd_post_kernel(const float* __restrict__ acc,
                                                       __nv_bfloat16* __restrict__ dq,
                                                       long long n8,
                                                       const float2* __restrict__ cs, int N,
                                                       int d) {
  const long long i0 = static_cast<long long>(blockIdx.x) * kPostThreads * kPostVecs + threadIdx.x;
  float4 a[kPostVecs], b[kPostVecs];
#pragma unroll
  for (int u = 0; u < kPostVecs; ++u) {
    const long long i = i0 + static_cast<long long>(u) * kPostThreads;
    if (i < n8) {
      a[u] = __ldg(reinterpret_cast<const float4*>(acc) + 2 * i);
      b[u] = __ldg(reinterpret_cast<const float4*>(acc) + 2 * i + 1);
    }
  }
  if (cs != nullptr) {
#pragma unroll
    for (int u = 0; u < kPostVecs; ++u) {
      const long long i = i0 + static_cast<long long>(u) * kPostThreads;
      if (i < n8) {
        const long long e = 8 * i;  // first element of the group; d % 8 == 0
        const long long row = e / d;
        const int col = static_cast<int>(e - row * d);
        const float2* t = cs + static_cast<size_t>(row % N) * (d / 2) + col / 2;
        rope_inv(a[u].x, a[u].y, __ldg(t));
        rope_inv(a[u].z, a[u].w, __ldg(t + 1));
        rope_inv(b[u].x, b[u].y, __ldg(t + 2));
        rope_inv(b[u].z, b[u].w, __ldg(t + 3));
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kPostVecs; ++u) {
    const long long i = i0 + static_cast<long long>(u) * kPostThreads;
    if (i < n8) {
      uint4 v;
      v.x = pack_bf16(a[u].x, a[u].y);
      v.y = pack_bf16(a[u].z, a[u].w);
      v.z = pack_bf16(b[u].x, b[u].y);
      v.w = pack_bf16(b[u].z, b[u].w);
      reinterpret_cast<uint4*>(dq)[i] = v;
    }
  }
}

// ---------------------------------------------------------------- main
template <int D>
struct BwdCfg {
  static constexpr int ES = 2;
  static constexpr int NBLK = D / 64;
  static constexpr int BLK_BYTES = kTile * 128;
  static constexpr int TILE_BYTES = NBLK * BLK_BYTES;
  static constexpr int QST = D == 64 ? 2 : 1;  // Q / dO ring depth
  static constexpr int NK_QK = D / 16;           // K-steps over d
  static constexpr int NK_T = kTile / 16;        // K-steps over 128 rows
  // tensor memory columns
  static constexpr int S_COL = 0, DP_COL = 128, DV_COL = 256;
  static constexpr int DK_COL = D == 64 ? 320 : 384;
  static constexpr int DQ_COL = D == 64 ? 384 : 128;  // d=128: shares dP's columns
  static constexpr int P_COL = D == 64 ? 448 : 0;     // d=128: shares S's columns
  static constexpr bool DQ_ALIAS_DP = D == 128;
  // shared memory (offsets from the 1024-B aligned base)
  static constexpr int OFF_K = 0, OFF_V = TILE_BYTES, OFF_Q = 2 * TILE_BYTES;
  static constexpr int OFF_DO = OFF_Q + QST * TILE_BYTES;
  static constexpr int OFF_DS = OFF_DO + QST * TILE_BYTES;  // 128x128 bf16, 2 blocks
  static constexpr int OFF_DQ = OFF_DS + 2 * BLK_BYTES;      // 2 fp32 boxes of 128x32
  static constexpr int OFF_L2 = OFF_DQ + 2 * BLK_BYTES;
  static constexpr int OFF_DSR = OFF_L2 + QST * 512;
  static constexpr int SMEM_BYTES = 1024 + OFF_DSR + QST * 512;
  static constexpr int THREADS = 512;
};

enum : int {
  C_KVFULL = 0, C_SFULL, C_DPFULL, C_PFULL, C_DSFULL, C_DSEMPTY, C_DQFULL, C_DQFREE, C_FINAL,
  C_DRAIN, C_DRAIN2, C_QFULL  // then QFULL[QST], DOFULL[QST], QEMPTY[QST]
};

// DQ = false: dK and dV only (the deterministic backward computes dQ in a
// kernel of its own, one CTA per query tile); no dQ MMA and no reductions.
template <int D, bool DQ>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1) bwd_main_kernel(const __grid_constant__ BwdArgs a) {
  using C = BwdCfg<D>;
  constexpr int QST = C::QST;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t bars[C_QFULL + 3 * QST];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = (a.N + kTile - 1) / kTile;  // the last tile may be partial
  const int BG = a.B * a.Hkv;
  const int G = a.H / a.Hkv;
  const int lin = blockIdx.x;
  const int j = lin / BG;  // key tile; j = 0 has the most query tiles under the causal mask
  const int bg = lin % BG;
  const int b = bg / a.Hkv, g = bg % a.Hkv;
  const int i0 = a.causal ? j : 0;
  const int nI = T - i0;
  const int nsteps = G * nI;

  const uint32_t base = smem_u32(smem);
  const uint32_t sK = base + C::OFF_K, sV = base + C::OFF_V, sDS = base + C::OFF_DS,
                 sDQ = base + C::OFF_DQ;
  auto sQ = [&](int s) { return base + C::OFF_Q + s * C::TILE_BYTES; };
  auto sDO = [&](int s) { return base + C::OFF_DO + s * C::TILE_BYTES; };
  const float* l2_s = reinterpret_cast<const float*>(smem + C::OFF_L2);
  const float* dsr_s = reinterpret_cast<const float*>(smem + C::OFF_DSR);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  auto qfull = [&](int s) { return bar(C_QFULL + s); };
  auto dofull = [&](int s) { return bar(C_QFULL + QST + s); };
  auto qempty = [&](int s) { return bar(C_QFULL + 2 * QST + s); };
  volatile int* abort = &abort_sh;
  unsigned int* status = a.status;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    mbar_init(bar(C_KVFULL), 1);
    mbar_init(bar(C_SFULL), 1);
    mbar_init(bar(C_DPFULL), 1);
    mbar_init(bar(C_PFULL), 256);
    mbar_init(bar(C_DSFULL), 256);
    mbar_init(bar(C_DSEMPTY), 1);
    mbar_init(bar(C_DQFULL), 1);
    mbar_init(bar(C_DQFREE), 128);
    mbar_init(bar(C_FINAL), 2);  // one commit per MMA issuer
    mbar_init(bar(C_DRAIN), 1);
    mbar_init(bar(C_DRAIN2), 1);
    for (int s = 0; s < QST; ++s) {
      mbar_init(qfull(s), 1);
      mbar_init(dofull(s), 1);
      mbar_init(qempty(s), 2 + 8);  // one commit per MMA issuer + one arrive per compute warp
    }
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&a.tmQ);
    prefetch_tmap(&a.tmK);
    prefetch_tmap(&a.tmV);
    prefetch_tmap(&a.tmdO);
    prefetch_tmap(&a.tmdQacc);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  auto step_hi = [&](int n, int& h, int& i) {
    h = g * G + n / nI;
    i = i0 + n % nI;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int kvh = b * a.Hkv + g;
      mbar_expect_tx(bar(C_KVFULL), 2 * C::TILE_BYTES);
      for (int k = 0; k < C::NBLK; ++k) {
        tma_load_3d(sK + k * C::BLK_BYTES, &a.tmK, bar(C_KVFULL), k * 64, j * kTile, kvh);
        tma_load_3d(sV + k * C::BLK_BYTES, &a.tmV, bar(C_KVFULL), k * 64, j * kTile, kvh);
      }
      int issued = 0;
      bool ok = true;
      for (int n = 0; n < nsteps; ++n) {
        const int s = n % QST;
        if (n >= QST && !mbar_wait(qempty(s), ((n / QST) - 1) & 1, abort, 20, status)) {
          ok = false;
          break;
        }
        int h, i;
        step_hi(n, h, i);
        const int bh = b * a.H + h;
        // per-row terms live in the workspace padded to whole tiles per head
        const size_t row0 = (static_cast<size_t>(bh) * T + i) * kTile;
        mbar_expect_tx(qfull(s), C::TILE_BYTES + 512);
        for (int k = 0; k < C::NBLK; ++k)
          tma_load_3d(sQ(s) + k * C::BLK_BYTES, &a.tmQ, qfull(s), k * 64, i * kTile, bh);
        bulk_load(base + C::OFF_L2 + s * 512, a.lse2 + row0, 512, qfull(s));
        mbar_expect_tx(dofull(s), C::TILE_BYTES + 512);
        for (int k = 0; k < C::NBLK; ++k)
          tma_load_3d(sDO(s) + k * C::BLK_BYTES, &a.tmdO, dofull(s), k * 64, i * kTile, bh);
        bulk_load(base + C::OFF_DSR + s * 512, a.delta + row0, 512, dofull(s));
        issued = n + 1;
      }
      mbar_wait_drain(bar(C_KVFULL), 0, 21, status);
      if (!ok) {
        for (int n = issued - QST > 0 ? issued - QST : 0; n < issued; ++n) {
          mbar_wait_drain(qfull(n % QST), (n / QST) & 1, 21, status);
          mbar_wait_drain(dofull(n % QST), (n / QST) & 1, 21, status);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer A
    // S, dP and dV.  A tcgen05.mma chain issued by one thread advances at
    // about one instruction per ~130 cycles whatever N is, so the step's MMAs
    // are split between two issuing warps: A (here) and B (warp 2: dK, dQ).
    // Each issuer's tcgen05.commit tracks only its own MMAs; every hazard
    // between the two goes through an mbarrier.
    if (lane == 0) {
      constexpr uint32_t idS = make_idesc<MmaKind::kBF16>(128, 128, false, false);
      constexpr uint32_t idDV = make_idesc<MmaKind::kBF16>(128, D, false, true);
      auto issue_s = [&](int n) {  // S^T = K_j Q_i^T
        const int s = n % QST;
#pragma unroll
        for (int k = 0; k < C::NK_QK; ++k) {
          const uint32_t off = (k / 4) * C::BLK_BYTES + (k % 4) * 32;
          mma_ss<MmaKind::kBF16>(tmem + C::S_COL, sdesc_sw128(sK + off, 16, 1024),
                                 sdesc_sw128(sQ(s) + off, 16, 1024), idS, k > 0 ? 1u : 0u);
        }
        mma_commit(bar(C_SFULL));
      };
      auto issue_dp = [&](int n) {  // dP^T = V_j dO_i^T
        const int s = n % QST;
#pragma unroll
        for (int k = 0; k < C::NK_QK; ++k) {
          const uint32_t off = (k / 4) * C::BLK_BYTES + (k % 4) * 32;
          mma_ss<MmaKind::kBF16>(tmem + C::DP_COL, sdesc_sw128(sV + off, 16, 1024),
                                 sdesc_sw128(sDO(s) + off, 16, 1024), idS, k > 0 ? 1u : 0u);
        }
        mma_commit(bar(C_DPFULL));
      };
      auto wait_q = [&](int n, uint32_t id) {
        return mbar_wait(qfull(n % QST), (n / QST) & 1, abort, id, status);
      };
      auto wait_do = [&](int n, uint32_t id) {
        return mbar_wait(dofull(n % QST), (n / QST) & 1, abort, id, status);
      };
      bool ok = mbar_wait(bar(C_KVFULL), 0, abort, 22, status) && wait_q(0, 23);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        ok = wait_do(0, 24);
        if (ok) {
          tc_fence_after();
          issue_dp(0);
        }
      }
      for (int n = 0; ok && n < nsteps; ++n) {
        const int s = n % QST;
        // dV += P^T dO_i
        if (!mbar_wait(bar(C_PFULL), n & 1, abort, 26, status)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < C::NK_T; ++k)
          mma_ts<MmaKind::kBF16>(tmem + C::DV_COL, tmem + C::P_COL + k * 8,
                                 sdesc_sw128(sDO(s) + k * 16 * 128, C::BLK_BYTES, 1024), idDV,
                                 (n > 0 || k > 0) ? 1u : 0u);
        mma_commit(qempty(s));  // dO_i no longer read by A
        if (n + 1 == nsteps) break;
        // S_{n+1}: the compute warps have read S_n (PFULL_n)
        if (!wait_q(n + 1, 23)) break;
        tc_fence_after();
        issue_s(n + 1);
        // dP_{n+1}: the compute warps have read dP_n (DSFULL_n); with d = 128
        // dQ_n shares dP's columns and must have been drained (DQFREE_n)
        if (!wait_do(n + 1, 24) || !mbar_wait(bar(C_DSFULL), n & 1, abort, 25, status)) break;
        if (DQ && C::DQ_ALIAS_DP && !mbar_wait(bar(C_DQFREE), n & 1, abort, 25, status)) break;
        tc_fence_after();
        issue_dp(n + 1);
      }
      mma_commit(bar(C_FINAL));
      mma_commit(bar(C_DRAIN));
      mbar_wait_drain(bar(C_DRAIN), 0, 29, status);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ MMA issuer B
    // dK and dQ.
    if (lane == 0) {
      constexpr uint32_t idDK = make_idesc<MmaKind::kBF16>(128, D, false, true);
      constexpr uint32_t idDQ = make_idesc<MmaKind::kBF16>(128, D, true, true);
      bool ok = mbar_wait(bar(C_KVFULL), 0, abort, 37, status);
      for (int n = 0; ok && n < nsteps; ++n) {
        const int s = n % QST;
        // dK += dS^T Q_i
        if (!mbar_wait(qfull(s), (n / QST) & 1, abort, 38, status) ||
            !mbar_wait(bar(C_DSFULL), n & 1, abort, 27, status))
          break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < C::NK_T; ++k) {
          const uint32_t off = (k / 4) * C::BLK_BYTES + (k % 4) * 32;
          mma_ss<MmaKind::kBF16>(tmem + C::DK_COL, sdesc_sw128(sDS + off, 16, 1024),
                                 sdesc_sw128(sQ(s) + k * 16 * 128, C::BLK_BYTES, 1024), idDK,
                                 (n > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(qempty(s));  // Q_i no longer read by B
        if (DQ) {
          // dQ_i = dS K_j (the dQ warps have drained dQ_{n-1} when d = 64)
          if (!C::DQ_ALIAS_DP && n > 0 &&
              !mbar_wait(bar(C_DQFREE), (n - 1) & 1, abort, 28, status))
            break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < C::NK_T; ++k)
            mma_ss<MmaKind::kBF16>(tmem + C::DQ_COL,
                                   sdesc_sw128(sDS + k * 16 * 128, C::BLK_BYTES, 1024),
                                   sdesc_sw128(sK + k * 16 * 128, C::BLK_BYTES, 1024), idDQ,
                                   k > 0 ? 1u : 0u);
        }
        mma_commit(bar(C_DSEMPTY));
        if (DQ) mma_commit(bar(C_DQFULL));
      }
      mma_commit(bar(C_FINAL));
      mma_commit(bar(C_DRAIN2));
      mbar_wait_drain(bar(C_DRAIN2), 0, 39, status);
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ compute
    // Two warpgroups: half 0 owns query columns 0..63 of every step, half 1
    // columns 64..127.  Thread = key row kr (TMEM lane).
    const int half = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int kr = quad * 32 + lane;
    const int q0 = 64 * half;
    const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const float c = a.scale * kLog2e;
    bool ok = true;
    for (int n = 0; n < nsteps; ++n) {
      const int s = n % QST;
      const uint32_t ph = (n / QST) & 1;
      int h, i;
      step_hi(n, h, i);
      if (!mbar_wait_warp(qfull(s), ph, abort, 30, status) ||
          !mbar_wait_warp(bar(C_SFULL), n & 1, abort, 31, status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t u0[32], u1[32];
      tmem_ld32(trow + C::S_COL + q0, u0);
      tmem_ld32(trow + C::S_COL + q0 + 32, u1);
      tmem_ld_wait(u0);
      reg_fence(u1);
      const float* l2 = l2_s + s * 128 + q0;
      const bool diag = a.causal && i == j;
      // A key past N (zero-filled by TMA) must not take part: under the
      // causal mask it lies after every real query and is masked with the
      // diagonal; without it, it is masked here.  Padded queries have
      // L2 = +inf, so their P is already 0.
      const bool kdead = !a.causal && j * kTile + kr >= a.N;
      uint32_t pk[32];  // P^T row, bf16 pairs (query 2t in the low half)
      auto make_p = [&](const uint32_t (&u)[32], int c0) {
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const float2 lv = *reinterpret_cast<const float2*>(l2 + c0 + 2 * t);
          float p0 = ex2(fmaf(__uint_as_float(u[2 * t]), c, -lv.x));
          float p1 = ex2(fmaf(__uint_as_float(u[2 * t + 1]), c, -lv.y));
          if (diag) {
            if (q0 + c0 + 2 * t < kr) p0 = 0.f;
            if (q0 + c0 + 2 * t + 1 < kr) p1 = 0.f;
          }
          if (kdead) p0 = p1 = 0.f;
          pk[c0 / 2 + t] = pack_bf16(p0, p1);
        }
      };
      make_p(u0, 0);
      make_p(u1, 32);
      tmem_st32(trow + C::P_COL + q0 / 2, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C_PFULL));
      // dS^T = P^T o (scale dP^T - Ds)
      if (!mbar_wait_warp(dofull(s), ph, abort, 32, status) ||
          !mbar_wait_warp(bar(C_DPFULL), n & 1, abort, 33, status) ||
          (n > 0 && !mbar_wait_warp(bar(C_DSEMPTY), (n - 1) & 1, abort, 34, status))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t v0[32], v1[32];
      tmem_ld32(trow + C::DP_COL + q0, v0);
      tmem_ld32(trow + C::DP_COL + q0 + 32, v1);
      tmem_ld_wait(v0);
      reg_fence(v1);
      const float* dsr = dsr_s + s * 128 + q0;
      uint8_t* dsrow = smem + C::OFF_DS + half * C::BLK_BYTES + kr * 128;
      auto make_ds = [&](const uint32_t (&v)[32], int c0) {
        uint32_t o[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const int q = c0 + 2 * t;
          const uint32_t pp = pk[q / 2];
          const float p0 = __uint_as_float(pp << 16), p1 = __uint_as_float(pp & 0xffff0000u);
          const float2 dv = *reinterpret_cast<const float2*>(dsr + q);
          const float d0 = p0 * fmaf(__uint_as_float(v[2 * t]), a.scale, -dv.x);
          const float d1 = p1 * fmaf(__uint_as_float(v[2 * t + 1]), a.scale, -dv.y);
          o[t] = pack_bf16(d0, d1);
        }
        // 32 queries = 64 B = chunks c0/8 .. c0/8 + 3 of this 128-B row
#pragma unroll
        for (int t4 = 0; t4 < 4; ++t4) {
          const int chunk = c0 / 8 + t4;
          *reinterpret_cast<uint4*>(dsrow + ((chunk ^ (kr & 7)) << 4)) =
              make_uint4(o[4 * t4], o[4 * t4 + 1], o[4 * t4 + 2], o[4 * t4 + 3]);
        }
      };
      make_ds(v0, 0);
      make_ds(v1, 32);
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(bar(C_DSFULL));
      __syncwarp();
      if (lane == 0) mbar_arrive(qempty(s));
    }
    // epilogue: half 0 writes dV rows, half 1 writes dK rows of this key tile
    if (ok) ok = mbar_wait_warp(bar(C_FINAL), 0, abort, 35, status);
    if (ok) {
      tc_fence_after();
      const bool row_ok = j * kTile + kr < a.N;  // rows past N are not stored
      const size_t row =
          (static_cast<size_t>(b) * a.Hkv + g) * a.N + static_cast<size_t>(j) * kTile + kr;
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(half == 0 ? a.dV : a.dK) + row * D;
      const uint32_t col = half == 0 ? C::DV_COL : C::DK_COL;
#pragma unroll
      // dK of rotated keys -> dK of the caller's keys (RoPE)
      const float2* rcs = (half == 1 && row_ok && a.rope_cs != nullptr)
                              ? a.rope_cs + static_cast<size_t>(j * kTile + kr) * (D / 2)
                              : nullptr;
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
  } else if (DQ && warp >= 12) {
    // ------------------------------------------------------------ dQ
    const int quad = warp & 3;
    const int qr = quad * 32 + lane;  // query row == TMEM lane of the dQ tile
    const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const bool leader = warp == 12 && lane == 0;
    for (int n = 0; n < nsteps; ++n) {
      int h, i;
      step_hi(n, h, i);
      const int bh = b * a.H + h;
      // the whole warpgroup unwinds together: it meets at named barriers below
      if (!named_bar_and(2, 128, mbar_wait_warp(bar(C_DQFULL), n & 1, abort, 36, status))) break;
      tc_fence_after();
#pragma unroll
      for (int hh = 0; hh < D / 64; ++hh) {
        uint32_t v0[32], v1[32];
        tmem_ld32(trow + C::DQ_COL + 64 * hh, v0);
        tmem_ld32(trow + C::DQ_COL + 64 * hh + 32, v1);
        tmem_ld_wait(v0);
        reg_fence(v1);
        if (hh == D / 64 - 1) {
          tc_fence_before();
          mbar_arrive(bar(C_DQFREE));
        }
        // staging free once the previous reduction has read it
        if (leader) bulk_wait_read0();
        named_bar_sync(2, 128);
#pragma unroll
        for (int box = 0; box < 2; ++box) {
          const uint32_t(&v)[32] = box == 0 ? v0 : v1;
          uint8_t* rowp = smem + C::OFF_DQ + box * C::BLK_BYTES + qr * 128;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            *reinterpret_cast<uint4*>(rowp + ((ch ^ (qr & 7)) << 4)) =
                make_uint4(v[4 * ch], v[4 * ch + 1], v[4 * ch + 2], v[4 * ch + 3]);
        }
        fence_proxy_async();
        named_bar_sync(2, 128);
        if (leader) {
          for (int box = 0; box < 2; ++box)
            tma_reduce_add_3d(&a.tmdQacc, sDQ + box * C::BLK_BYTES, 64 * hh + 32 * box,
                              i * kTile, bh);
          bulk_commit();
        }
      }
    }
    if (leader) bulk_wait0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}


template <int D, bool DQ>
cudaError_t launch_main_t(const BwdArgs& a, cudaStream_t stream) {
  using C = BwdCfg<D>;
  auto kern = bwd_main_kernel<D, DQ>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(a.B) * a.Hkv * ((a.N + kTile - 1) / kTile);
  kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_pre(const BwdArgs& a, cudaStream_t stream) {
  const int npad = (a.N + kTile - 1) / kTile * kTile;
  const long long prows = static_cast<long long>(a.B) * a.H * npad;
  const int esize = a.dtype == 0 ? 2 : 4;
  const int tpr = a.d * esize / 16;
  const long long per_block = static_cast<long long>(kPreThreads / tpr) * kPreRows;  // divides 128
  const unsigned grid = static_cast<unsigned>((prows + per_block - 1) / per_block);
  if (a.dtype == 0 && a.d == 64)
    bwd_pre_kernel<__nv_bfloat16, 64><<<grid, kPreThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(a.O), static_cast<const __nv_bfloat16*>(a.dO), a.lse,
        a.delta, a.lse2, a.dq_acc, prows, a.N, npad, a.scale);
  else if (a.dtype == 0 && a.d == 128)
    bwd_pre_kernel<__nv_bfloat16, 128><<<grid, kPreThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(a.O), static_cast<const __nv_bfloat16*>(a.dO), a.lse,
        a.delta, a.lse2, a.dq_acc, prows, a.N, npad, a.scale);
  else if (a.dtype == 1 && a.d == 64)
    bwd_pre_kernel<float, 64><<<grid, kPreThreads, 0, stream>>>(
        static_cast<const float*>(a.O), static_cast<const float*>(a.dO), a.lse, a.delta, a.lse2,
        a.dq_acc, prows, a.N, npad, a.scale);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_bwd_main(const BwdArgs& a, cudaStream_t stream) {
  if (a.dtype == 0 && a.d == 64)
    return a.deterministic ? launch_main_t<64, false>(a, stream) : launch_main_t<64, true>(a, stream);
  if (a.dtype == 0 && a.d == 128)
    return a.deterministic ? launch_main_t<128, false>(a, stream)
                           : launch_main_t<128, true>(a, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_post(const BwdArgs& a, cudaStream_t stream) {
  const long long n8 = static_cast<long long>(a.B) * a.H * a.N * a.d / 8;
  const long long per_block = static_cast<long long>(kPostThreads) * kPostVecs;
  bwd_post_kernel<<<static_cast<unsigned>((n8 + per_block - 1) / per_block), kPostThreads, 0,
                    stream>>>(
      a.dq_acc, static_cast<__nv_bfloat16*>(a.dQ), n8, a.rope_cs, a.N, a.d);
  return cudaGetLastError();
}

}  // namespace nea
