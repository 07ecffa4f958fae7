// bwd.cu -- causal grouped-query FlashAttention backward on tcgen05 / TMEM.
//
// "NanoEuler: Hand-writing GPT-2 in Pure C/CUDA", section "Hand-written
// Backpropagation": every gradient is derived and written by hand.  For
// softmax attention with upstream dO:
//   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),  D = rowsum(dO o O),
//   dQ = scale dS K,  dK = scale dS^T Q,  P recomputed from the saved LSE.
//
// Three kernels:
//  bwd_pre   (HBM-bound)  Ds = scale * rowsum(dO o O), NL2 = -LSE * log2(e),
//                         and zeroes the fp32 dQ accumulator;
//  bwd_main  one CTA per (batch, KV head, 128-row key tile j); it walks the
//            group's query heads and the query tiles i >= j (causal):
//              warp 0      TMA producer (K_j, V_j once; Q_i, dO_i, NL2_i, Ds_i
//                          per step into a ring), and MMA issuer of
//                          dQ' = dS' K (SS, A and B MN-major; the same smem
//                          bytes as dS'^T), interleaved without blocking
//              warp 1      MMA issuer: S^T = K Q^T, dP^T = V dO^T (SS);
//                          owns the TMEM allocation
//              warp 2      MMA issuer: dV += P^T dO (TS, P^T from TMEM)
//              warp 3      MMA issuer: dK' += dS'^T Q (SS, B MN-major)
//              warps 4..19 "compute", four groups of four warps splitting
//                          the 128 query columns: thread = key row;
//                          P^T = exp2(S^T c + NL2) to TMEM (bf16),
//                          dS'^T = P^T o (Ds - scale dP^T) to smem (bf16,
//                          128-B swizzle, two buffers at d = 64)
//              warps 20..23 dQ drain (thread = query row): dQ' TMEM ->
//                          smem -> TMA reduce-add (fp32) into the accumulator
//            dK and dV stay in TMEM for the whole CTA: the sum over the
//            group's query heads needs no atomics.
//  bwd_post  dQ = bf16(-accumulator).
#include <algorithm>

#include "nea_internal.h"
#include "ptx.cuh"
#include "rope.cuh"
#include "trace.cuh"

namespace nea {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

#ifdef NEA_TRACE
// Timeline of CTA 0 of the main kernel (the longest one under the causal
// mask): rows 0 producer, 1 / 2 MMA issuers, 3 / 4 first warp of each compute
// warpgroup, 5 first dQ warp.
__device__ long long g_trace_bwd[kTraceRoles * kTraceEvents];
// Every CTA of the main kernel: (start, end) in global nanoseconds and its SM.
constexpr int kTraceCtas = 4096;
__device__ long long g_trace_cta[3 * kTraceCtas];
__device__ __forceinline__ long long global_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ int sm_id() {
  int v;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(v));
  return v;
}
#define NEA_TRACE_BASE g_trace_bwd
#else
#define NEA_TRACE_BASE nullptr
#endif

// ---------------------------------------------------------------- preprocess
// Walks the per-head rows padded to whole 128-row tiles (npad = T * 128):
// padded row p = bh * npad + n.  Real rows (n < N) get Ds = scale * dO.O and
// NL2 = -LSE * log2(e); padding rows get Ds = 0 and NL2 = -inf, so that the
// backward kernels' exp2(S c + NL2) is exactly 0 for them.  TPR threads per
// row, each owning 16 bytes of O and dO.  A unit of work is kPreRows passes
// of a block's rows (a divisor of a 128-row tile); every thread issues all
// loads of its unit (the rows' LSE included) before any use.
constexpr int kPreRows = 4;
constexpr int kPreThreads = 256;

// Row terms of the main kernel's S and dP accumulators, as one K row of a
// K = 16 MMA operand: x = hi + mid + lo in bf16 (each part the rounded
// remainder of the previous ones), then zeros.  Only the first 16 bytes of
// each row (K elements 0..7) are stored, row-major: 16 bytes per query row,
// 2 KB per 128-row tile; the main kernel keeps the zero half in shared
// memory.
__device__ __forceinline__ void write_fold_row(uint16_t* tile, int q, float x) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(hi);
  const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
  const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
  uint4 v0;
  v0.x = static_cast<uint32_t>(__bfloat16_as_ushort(hi)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(mid)) << 16);
  v0.y = static_cast<uint32_t>(__bfloat16_as_ushort(lo));
  v0.z = v0.w = 0u;
  *reinterpret_cast<uint4*>(tile + q * 8) = v0;
}

template <typename T, int D>
__global__ void __launch_bounds__(kPreThreads) bwd_pre_kernel(const T* __restrict__ O,
                                                      const T* __restrict__ dO,
                                                      const float* __restrict__ lse,
                                                      float* __restrict__ ds_row,
                                                      float* __restrict__ l2_row,
                                                      float* __restrict__ dq_acc,
                                                      uint16_t* __restrict__ fold, long long prows,
                                                      int N, int npad, float scale) {
  constexpr int EPV = 16 / sizeof(T);  // elements per 16-B vector
  constexpr int TPR = D / EPV;         // threads per row
  constexpr int RPB = kPreThreads / TPR;  // rows per block per pass
  constexpr int UNIT = RPB * kPreRows;    // rows per unit
  static_assert(kTile % UNIT == 0, "a unit's rows must divide a tile");
  const int sub = threadIdx.x % TPR;
  const long long units = prows / UNIT;
  for (long long unit = blockIdx.x; unit < units; unit += gridDim.x) {
    // A unit lies inside one head: bh and the row offset are unit-uniform.
    const long long pb = unit * UNIT;
    const long long bh = pb / npad;
    const int nb = static_cast<int>(pb - bh * npad) + threadIdx.x / TPR;
    const long long p0 = pb + threadIdx.x / TPR;
    uint4 ov[kPreRows], gv[kPreRows];
    float lv[kPreRows];
    long long rrow[kPreRows];  // unpadded row index, or -1 for padding
#pragma unroll
    for (int u = 0; u < kPreRows; ++u) {
      const int n = nb + u * RPB;
      rrow[u] = n < N ? bh * N + n : -1;
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
      if (sub == 0) {
        ds_row[p] = rrow[u] >= 0 ? acc * scale : 0.f;
        l2_row[p] = rrow[u] >= 0 ? -lv[u] * kLog2e : -INFINITY;
        if (fold != nullptr) {
          // tile pair p / 128 = (head, query tile): S' = S - LSE / scale
          // (padding: -1e30, so that P = 0 there), then dP' = dP - D
          uint16_t* tile = fold + (p / kTile) * 2048;
          const int q = static_cast<int>(p % kTile);
          write_fold_row(tile, q, rrow[u] >= 0 ? -lv[u] / scale : -1e30f);
          write_fold_row(tile + 1024, q, rrow[u] >= 0 ? -acc : 0.f);
        }
      }
      // zero this thread's share of the fp32 accumulator row (D floats)
      if (dq_acc != nullptr && rrow[u] >= 0) {
        float4* z = reinterpret_cast<float4*>(dq_acc + static_cast<size_t>(rrow[u]) * D);
#pragma unroll
        for (int k = sub; k < D / 4; k += TPR) z[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
}

// ---------------------------------------------------------------- dQ cast
// Each thread converts kPostVecs groups of 8 fp32 -> 8 bf16 per round.  The
// main kernel accumulates -dQ (see
// its sign convention), so the cast negates.  With a RoPE table, the 4 pairs
// of a group are first turned back by their row's angles.
constexpr int kPostVecs = 4;
constexpr int kPostThreads = 256;

__global__ void __launch_bounds__(kPostThreads) bwd_post_kernel(const float* __restrict__ acc,
                                                       __nv_bfloat16* __restrict__ dq,
                                                       long long n8,
                                                       const float2* __restrict__ cs, int N,
                                                       int d) {
  const long long per_round = static_cast<long long>(gridDim.x) * kPostThreads * kPostVecs;
  for (long long i0 = static_cast<long long>(blockIdx.x) * kPostThreads * kPostVecs + threadIdx.x;
       i0 < n8; i0 += per_round) {
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
        v.x = pack_bf16(-a[u].x, -a[u].y);
        v.y = pack_bf16(-a[u].z, -a[u].w);
        v.z = pack_bf16(-b[u].x, -b[u].y);
        v.w = pack_bf16(-b[u].z, -b[u].w);
        reinterpret_cast<uint4*>(dq)[i] = v;
      }
    }
  }
}

// ---------------------------------------------------------------- main
template <int D>
struct BwdCfg {
  static constexpr int NBLK = D / 64;
  static constexpr int BLK_BYTES = kTile * 128;
  static constexpr int TILE_BYTES = NBLK * BLK_BYTES;
  // Ring depths.  Q_n is read by S_n and by dK_n, which can only start once
  // dS'_n is formed, so Q stages are held the longest; dO_n is read by dP_n
  // and dV_n and freed earlier.
  static constexpr int QST = D == 64 ? 3 : 1;   // Q ring depth
  static constexpr int DOST = D == 64 ? 2 : 1;  // dO ring depth
  static constexpr int DSST = D == 64 ? 2 : 1;  // dS^T buffers in shared memory
  static constexpr int NK_QK = D / 16;          // K-steps over d
  static constexpr int NK_T = kTile / 16;       // K-steps over 128 rows
  // tensor memory columns
  static constexpr int S_COL = 0, DP_COL = 128, DV_COL = 256;
  static constexpr int DK_COL = D == 64 ? 320 : 384;
  static constexpr int DQ_COL = D == 64 ? 384 : 128;  // d=128: shares dP's columns
  // Compute warps: NGRP groups of four (one warp per TMEM lane quadrant),
  // group q owns query columns [32 q, 32 q + 32) of every step.
  static constexpr int NGRP = 4;
  static constexpr int NCW = 4 * NGRP;  // compute warps
  // P^T as packed bf16: group q writes its 32 queries (16 columns) inside
  // its own S^T columns, which it has already read (P_COL + q * P_GSTRIDE).
  static constexpr int P_COL = 0;
  static constexpr int P_GSTRIDE = 32;
  static constexpr bool DQ_ALIAS_DP = D == 128;
  static constexpr bool P_ALIAS_S = true;
  // d = 64: dS'^T also goes to tensor memory (packed bf16, group q at
  // DST_COL + 16 q), so that dK is a TS MMA and reads only Q from shared
  // memory.  d = 128 has no columns left: dK reads dS'^T from shared memory.
  static constexpr bool DK_TS = D == 64;
  static constexpr int DST_COL = 448;
  // shared memory (offsets from the 1024-B aligned base)
  static constexpr int OFF_K = 0, OFF_V = TILE_BYTES, OFF_Q = 2 * TILE_BYTES;
  static constexpr int OFF_DO = OFF_Q + QST * TILE_BYTES;
  static constexpr int OFF_DS = OFF_DO + DOST * TILE_BYTES;  // DSST x (128x128 bf16, 2 blocks)
  static constexpr int OFF_DQ = OFF_DS + DSST * 2 * BLK_BYTES;  // one fp32 box of 128x32
  // K = 16 operands of the row-term MMAs (4 KB each): the ones tile, and per
  // ring stage the query tile's -LSE/scale (with Q) and -D (with dO) tiles.
  // Each holds K elements 0..7 of its 128 rows in its first 2 KB (row r at
  // r * 16) and zeros (K elements 8..15) in the second: the no-swizzle
  // K-major layout with core matrices 128 B apart along M/N, 2 KB along K.
  static constexpr int FOLD_BYTES = 4096;
  static constexpr int OFF_ONES = OFF_DQ + BLK_BYTES;
  static constexpr int OFF_FU = OFF_ONES + FOLD_BYTES;
  static constexpr int OFF_FW = OFF_FU + QST * FOLD_BYTES;
  static constexpr int SMEM_BYTES = 1024 + OFF_FW + DOST * FOLD_BYTES;
  // warps 0..3 producer (+ dQ issuer) and issuers, 4..4+NCW-1 compute,
  // then 4 dQ drain warps
  static constexpr int DQ_WARP0 = 4 + NCW;
  static constexpr int THREADS = 32 * (DQ_WARP0 + 4);
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

// mbarrier slots.  Per step n (tile pair of key tile j and one query tile):
//   SFULL / DPFULL  S^T_n / dP^T_n are in tensor memory (issuer 1)
//   SFREE / DPFREE  the compute warps have read them (next S / dP may overwrite)
//   PFULL           P^T_n is in tensor memory (compute warps)
//   PFREE           dV += P^T_n dO_n is done (the next P may overwrite)
//   DSFULL[b]       dS^T_n is in shared-memory buffer b = n % DSST
//   DSEMPTY[b]      dK and dQ have read buffer b
//   DQFULL          dQ_n is in tensor memory; DQFREE: the dQ warps have read it
//   DKDONE          dK += dS'^T_n Q_n is done (the next dS'^T may overwrite TMEM)
//   QFULL / QEMPTY [n % QST]      ring stage of Q_n (and the -LSE/scale tile)
//   DOFULL / DOEMPTY [n % DOST]   ring stage of dO_n (and the -D tile)
enum : int {
  C_KVFULL = 0, C_SFULL, C_SFREE, C_DPFULL, C_DPFREE, C_PFULL, C_PFREE, C_DQFULL, C_DQFREE,
  C_DKDONE, C_FINAL, C_DRAIN1, C_DRAIN2, C_DRAIN3, C_DRAIN4,
  C_DSFULL  // then DSFULL[DSST], DSEMPTY[DSST],
                                                              // QFULL[QST], QEMPTY[QST],
                                                              // DOFULL[DOST], DOEMPTY[DOST]
};

// DQ = false: dK and dV only (the deterministic backward computes dQ in a
// kernel of its own, one CTA per query tile); no dQ MMA and no reductions.
//
// Sign convention: the compute warps form dS'^T = P^T o (Ds - scale dP^T)
// = -scale dS^T (one packed FMA with a negative constant), so the dK
// accumulator holds -dK (negated in the epilogue) and the dQ partials add up
// to -dQ (negated by the cast kernel).
template <int D, bool DQ>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1) bwd_main_kernel(const __grid_constant__ BwdArgs a) {
  using C = BwdCfg<D>;
  constexpr int QST = C::QST, DOST = C::DOST, DSST = C::DSST;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t bars[C_DSFULL + 2 * DSST + 2 * QST + 2 * DOST];
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
  const uint32_t sK = base + C::OFF_K, sV = base + C::OFF_V, sDQ = base + C::OFF_DQ;
  auto sQ = [&](int s) { return base + C::OFF_Q + s * C::TILE_BYTES; };
  auto sDO = [&](int s) { return base + C::OFF_DO + s * C::TILE_BYTES; };
  auto sDS = [&](int bb) { return base + C::OFF_DS + bb * 2 * C::BLK_BYTES; };
  const uint32_t sONES = base + C::OFF_ONES;
  auto sFU = [&](int s) { return base + C::OFF_FU + s * C::FOLD_BYTES; };
  auto sFW = [&](int s) { return base + C::OFF_FW + s * C::FOLD_BYTES; };
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  auto dsfull = [&](int bb) { return bar(C_DSFULL + bb); };
  auto dsempty = [&](int bb) { return bar(C_DSFULL + DSST + bb); };
  auto qfull = [&](int s) { return bar(C_DSFULL + 2 * DSST + s); };
  auto qempty = [&](int s) { return bar(C_DSFULL + 2 * DSST + QST + s); };
  auto dofull = [&](int s) { return bar(C_DSFULL + 2 * DSST + 2 * QST + s); };
  auto doempty = [&](int s) { return bar(C_DSFULL + 2 * DSST + 2 * QST + DOST + s); };
  volatile int* abort = &abort_sh;
  unsigned int* status = a.status;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    mbar_init(bar(C_KVFULL), 1);
    mbar_init(bar(C_SFULL), 1);
    mbar_init(bar(C_SFREE), C::NCW);  // one arrive per compute warp
    mbar_init(bar(C_DPFULL), 1);
    mbar_init(bar(C_DPFREE), C::NCW);
    mbar_init(bar(C_PFULL), C::NCW);
    mbar_init(bar(C_PFREE), 1);
    mbar_init(bar(C_DQFULL), 1);
    mbar_init(bar(C_DQFREE), 4);  // one arrive per dQ warp
    mbar_init(bar(C_DKDONE), 1);
    mbar_init(bar(C_FINAL), 2);   // the dV and dK issuers' last commits
    mbar_init(bar(C_DRAIN1), 1);
    mbar_init(bar(C_DRAIN2), 1);
    mbar_init(bar(C_DRAIN3), 1);
    mbar_init(bar(C_DRAIN4), 1);
    for (int bb = 0; bb < DSST; ++bb) {
      mbar_init(dsfull(bb), C::NCW);
      mbar_init(dsempty(bb), DQ ? 2 : 1);  // the dK and dQ issuers
    }
    for (int s = 0; s < QST; ++s) {
      mbar_init(qfull(s), 1);
      mbar_init(qempty(s), 2);  // read by S (issuer 1) and dK (issuer 3)
    }
    for (int s = 0; s < DOST; ++s) {
      mbar_init(dofull(s), 1);
      mbar_init(doempty(s), 2);  // read by dP (issuer 1) and dV (issuer 2)
    }
    fence_barrier_init();
    // The CTA's first loads go out now, before the TMEM allocation and the
    // shared-memory setup below: K_j and V_j, and the first ring stages of
    // Q and dO with their row-term tiles (the producer loop continues from
    // there).  Their latency is most of a short CTA's fixed cost.
    prefetch_tmap(&a.tmQ);
    prefetch_tmap(&a.tmK);
    prefetch_tmap(&a.tmV);
    prefetch_tmap(&a.tmdO);
    prefetch_tmap(&a.tmdQacc);
    const int kvh = b * a.Hkv + g;
    mbar_expect_tx(bar(C_KVFULL), 2 * C::TILE_BYTES);
    for (int k = 0; k < C::NBLK; ++k) {
      tma_load_3d(sK + k * C::BLK_BYTES, &a.tmK, bar(C_KVFULL), k * 64, j * kTile, kvh);
      tma_load_3d(sV + k * C::BLK_BYTES, &a.tmV, bar(C_KVFULL), k * 64, j * kTile, kvh);
    }
    for (int n = 0; n < QST && n < nsteps; ++n) {
      const int h = g * G + n / nI, i = i0 + n % nI, bh = b * a.H + h;
      const uint16_t* fold = a.fold + (static_cast<size_t>(bh) * T + i) * 2048;
      mbar_expect_tx(qfull(n), C::TILE_BYTES + 2048);
      for (int k = 0; k < C::NBLK; ++k)
        tma_load_3d(sQ(n) + k * C::BLK_BYTES, &a.tmQ, qfull(n), k * 64, i * kTile, bh);
      bulk_load(sFU(n), fold, 2048, qfull(n));
    }
    for (int n = 0; n < DOST && n < nsteps; ++n) {
      const int h = g * G + n / nI, i = i0 + n % nI, bh = b * a.H + h;
      const uint16_t* fold = a.fold + (static_cast<size_t>(bh) * T + i) * 2048;
      mbar_expect_tx(dofull(n), C::TILE_BYTES + 2048);
      for (int k = 0; k < C::NBLK; ++k)
        tma_load_3d(sDO(n) + k * C::BLK_BYTES, &a.tmdO, dofull(n), k * 64, i * kTile, bh);
      bulk_load(sFW(n), fold + 1024, 2048, dofull(n));
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), 512);
    tmem_relinquish();
  }
  // the ones operand of the row-term MMAs (every key row = (1, 1, 1, 0, ...,
  // 0)) and the zero halves of the ring's row-term tiles
  for (int c = threadIdx.x; c < (1 + QST + DOST) * 128; c += blockDim.x) {
    const int t = c / 128, r = c % 128;
    uint8_t* tile = smem + (t == 0 ? C::OFF_ONES : t <= QST ? C::OFF_FU + (t - 1) * C::FOLD_BYTES
                                                            : C::OFF_FW + (t - 1 - QST) * C::FOLD_BYTES);
    if (t == 0)
      *reinterpret_cast<uint4*>(tile + r * 16) = make_uint4(0x3F803F80u, 0x00003F80u, 0u, 0u);
    *reinterpret_cast<uint4*>(tile + 2048 + r * 16) = make_uint4(0u, 0u, 0u, 0u);
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  auto step_hi = [&](int n, int& h, int& i) {
    h = g * G + n / nI;
    i = i0 + n % nI;
  };
  // A-operand address of P^T for K-step k (16 queries) of the dV MMA.
  auto p_col = [&](int k) { return C::P_COL + (k / 2) * C::P_GSTRIDE + (k % 2) * 8; };

  const bool traced = blockIdx.x == 0 && lane == 0;
#ifdef NEA_TRACE
  if (threadIdx.x == 0 && blockIdx.x < kTraceCtas) {
    g_trace_cta[3 * blockIdx.x] = global_ns();
    g_trace_cta[3 * blockIdx.x + 2] = sm_id();
  }
#endif
  if (warp == 0) {
    // ------------------------------------------------------------ producer + dQ issuer
    // One warp runs two roles without blocking on either: it issues
    // dQ'_n = dS'_n K_j (A = the same shared-memory bytes as dS'^T, read
    // MN-major) as soon as dS'^T_n is in shared memory and the drain warps
    // have read dQ'_{n-1} out of TMEM, and it keeps the Q and dO rings
    // full.  The dQ MMAs go first: they are on the critical path, the loads
    // run ahead of their use.  The whole warp runs the loop (its tests are
    // warp-uniform); one elected lane issues the copies, MMAs and commits.
    {
      Tracer tr(NEA_TRACE_BASE, traced, 0);
      Tracer trq(NEA_TRACE_BASE, traced, 7);
      tr.ev(0);
      constexpr uint32_t idDQ = make_idesc<MmaKind::kBF16>(128, D, true, true);
      // next step to load Q / dO for (the prologue issued the first stages),
      // and to issue dQ for
      int nl = QST < nsteps ? QST : nsteps, nd = DOST < nsteps ? DOST : nsteps;
      int nq = DQ ? 0 : nsteps;
      bool ok = true;
      long long idle0 = clock64();
      while (nl < nsteps || nd < nsteps || nq < nsteps) {
        bool progress = false;
        if (nq < nsteps) {
          const int bb = nq % DSST;
          if (mbar_test_warp(dsfull(bb), (nq / DSST) & 1) &&
              (nq == 0 || mbar_test_warp(bar(C_DQFREE), (nq - 1) & 1))) {
            trq.ev(22);
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
              for (int k = 0; k < C::NK_T; ++k)
                mma_ss<MmaKind::kBF16>(tmem + C::DQ_COL,
                                       sdesc_sw128(sDS(bb) + k * 16 * 128, C::BLK_BYTES, 1024),
                                       sdesc_sw128(sK + k * 16 * 128, C::BLK_BYTES, 1024), idDQ,
                                       k > 0 ? 1u : 0u);
              mma_commit(dsempty(bb));
              mma_commit(bar(C_DQFULL));
            }
            __syncwarp();
            trq.ev(23);
            ++nq;
            progress = true;
          }
        }
        // the two row-term tiles of (head, query tile): 2 KB each in the workspace
        if (nl < nsteps) {
          const int s = nl % QST;
          if (nl < QST || mbar_test_warp(qempty(s), ((nl / QST) - 1) & 1)) {
            int h, i;
            step_hi(nl, h, i);
            const int bh = b * a.H + h;
            const uint16_t* fold = a.fold + (static_cast<size_t>(bh) * T + i) * 2048;
            if (elect_one()) {
              mbar_expect_tx(qfull(s), C::TILE_BYTES + 2048);
              for (int k = 0; k < C::NBLK; ++k)
                tma_load_3d(sQ(s) + k * C::BLK_BYTES, &a.tmQ, qfull(s), k * 64, i * kTile, bh);
              bulk_load(sFU(s), fold, 2048, qfull(s));
            }
            __syncwarp();
            tr.ev(1);
            ++nl;
            progress = true;
          }
        }
        if (nd < nsteps) {
          const int s = nd % DOST;
          if (nd < DOST || mbar_test_warp(doempty(s), ((nd / DOST) - 1) & 1)) {
            int h, i;
            step_hi(nd, h, i);
            const int bh = b * a.H + h;
            const uint16_t* fold = a.fold + (static_cast<size_t>(bh) * T + i) * 2048;
            if (elect_one()) {
              mbar_expect_tx(dofull(s), C::TILE_BYTES + 2048);
              for (int k = 0; k < C::NBLK; ++k)
                tma_load_3d(sDO(s) + k * C::BLK_BYTES, &a.tmdO, dofull(s), k * 64, i * kTile, bh);
              bulk_load(sFW(s), fold + 1024, 2048, dofull(s));
            }
            __syncwarp();
            ++nd;
            progress = true;
          }
        }
        if (progress) {
          idle0 = clock64();
          continue;
        }
        // nothing ready: back off briefly; give up with the other roles
        // (lane 0 decides for the warp)
        int give_up = 0;
        if (lane == 0) {
          if (*abort) {
            give_up = 1;
          } else if (clock64() - idle0 > kWaitCycles) {
            *abort = 1;
            atomicOr(status, kStatusTimeout | (20u << 8));
            give_up = 1;
          }
        }
        if (__shfl_sync(0xffffffffu, give_up, 0)) {
          ok = false;
          break;
        }
        __nanosleep(32);
      }
      // everything this warp started must finish before the CTA exits: its
      // MMAs, and (when unwinding) the loads it issued
      if (elect_one()) mma_commit(bar(C_DRAIN4));
      __syncwarp();
      mbar_wait_drain(bar(C_DRAIN4), 0, 41, status);
      mbar_wait_drain(bar(C_KVFULL), 0, 21, status);
      if (!ok) {
        for (int n = nl - QST > 0 ? nl - QST : 0; n < nl; ++n)
          mbar_wait_drain(qfull(n % QST), (n / QST) & 1, 21, status);
        for (int n = nd - DOST > 0 ? nd - DOST : 0; n < nd; ++n)
          mbar_wait_drain(dofull(n % DOST), (n / DOST) & 1, 21, status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ issuer 1: S^T, dP^T
    // The five GEMMs of a step are spread over four issuing warps (S^T and
    // dP^T here; dV, dK and dQ each on a warp of its own), so that the
    // tensor core always has work queued.  Every hazard between issuers
    // goes through an mbarrier.  Each issuing warp runs its loop converged
    // (warp-uniform waits) and issues from one elected lane.
    {
      Tracer tr(NEA_TRACE_BASE, traced, 1);
      constexpr uint32_t idS = make_idesc<MmaKind::kBF16>(128, 128, false, false);
      bool ok = mbar_wait_warp(bar(C_KVFULL), 0, abort, 22, status);
      for (int n = 0; ok && n < nsteps; ++n) {
        const int s = n % QST, sd = n % DOST;
        const uint32_t ph = (n / QST) & 1, phd = (n / DOST) & 1;
        // S^T_n = K_j Q_i^T: Q_n has landed; the compute warps have read S^T_{n-1}
        // (and, with P in S's columns, dV_{n-1} has read P^T_{n-1})
        ok = mbar_wait_warp(qfull(s), ph, abort, 23, status) &&
             (n == 0 || mbar_wait_warp(bar(C_SFREE), (n - 1) & 1, abort, 24, status)) &&
             (!C::P_ALIAS_S || n == 0 ||
              mbar_wait_warp(bar(C_PFREE), (n - 1) & 1, abort, 24, status));
        if (!ok) break;
        tr.ev(12);
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < C::NK_QK; ++k) {
            const uint32_t off = (k / 4) * C::BLK_BYTES + (k % 4) * 32;
            mma_ss<MmaKind::kBF16>(tmem + C::S_COL, sdesc_sw128(sK + off, 16, 1024),
                                   sdesc_sw128(sQ(s) + off, 16, 1024), idS, k > 0 ? 1u : 0u);
          }
          // S'^T = S^T + 1 u^T, u = -LSE / scale of each query (one K = 16 step)
          mma_ss<MmaKind::kBF16>(tmem + C::S_COL, sdesc_k16(sONES), sdesc_k16(sFU(s)), idS, 1u);
          mma_commit(bar(C_SFULL));
          mma_commit(qempty(s));  // Q_n no longer read by this issuer
        }
        __syncwarp();
        tr.ev(13);
        // dP^T_n = V_j dO_i^T: dO_n has landed; dP^T_{n-1} has been read (and,
        // with dQ in dP's columns, dQ_{n-1} has been drained)
        ok = mbar_wait_warp(dofull(sd), phd, abort, 25, status) &&
             (n == 0 || mbar_wait_warp(bar(C_DPFREE), (n - 1) & 1, abort, 25, status)) &&
             (!(DQ && C::DQ_ALIAS_DP) || n == 0 ||
              mbar_wait_warp(bar(C_DQFREE), (n - 1) & 1, abort, 25, status));
        if (!ok) break;
        tr.ev(14);
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < C::NK_QK; ++k) {
            const uint32_t off = (k / 4) * C::BLK_BYTES + (k % 4) * 32;
            mma_ss<MmaKind::kBF16>(tmem + C::DP_COL, sdesc_sw128(sV + off, 16, 1024),
                                   sdesc_sw128(sDO(sd) + off, 16, 1024), idS, k > 0 ? 1u : 0u);
          }
          // dP'^T = dP^T - 1 D^T (one K = 16 step)
          mma_ss<MmaKind::kBF16>(tmem + C::DP_COL, sdesc_k16(sONES), sdesc_k16(sFW(sd)), idS, 1u);
          mma_commit(bar(C_DPFULL));
          mma_commit(doempty(sd));  // dO_n no longer read by this issuer
        }
        __syncwarp();
        tr.ev(15);
      }
      if (elect_one()) mma_commit(bar(C_DRAIN1));
      __syncwarp();
      mbar_wait_drain(bar(C_DRAIN1), 0, 29, status);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ issuer 2: dV
    {
      Tracer tr(NEA_TRACE_BASE, traced, 2);
      constexpr uint32_t idDV = make_idesc<MmaKind::kBF16>(128, D, false, true);
      bool ok = true;
      for (int n = 0; ok && n < nsteps; ++n) {
        const int s = n % DOST;
        // dV += P^T_n dO_n (P^T from tensor memory)
        ok = mbar_wait_warp(dofull(s), (n / DOST) & 1, abort, 26, status) &&
             mbar_wait_warp(bar(C_PFULL), n & 1, abort, 26, status);
        if (!ok) break;
        tr.ev(10);
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < C::NK_T; ++k)
            mma_ts<MmaKind::kBF16>(tmem + C::DV_COL, tmem + p_col(k),
                                   sdesc_sw128(sDO(s) + k * 16 * 128, C::BLK_BYTES, 1024), idDV,
                                   (n > 0 || k > 0) ? 1u : 0u);
          mma_commit(bar(C_PFREE));
          mma_commit(doempty(s));
        }
        __syncwarp();
        tr.ev(11);
      }
      if (elect_one()) {
        mma_commit(bar(C_FINAL));
        mma_commit(bar(C_DRAIN2));
      }
      __syncwarp();
      mbar_wait_drain(bar(C_DRAIN2), 0, 39, status);
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ issuer 3: dK
    {
      Tracer tr(NEA_TRACE_BASE, traced, 3);
      constexpr uint32_t idDK = make_idesc<MmaKind::kBF16>(128, D, false, true);
      bool ok = true;
      for (int n = 0; ok && n < nsteps; ++n) {
        const int s = n % QST, bb = n % DSST;
        // dK' += dS'^T_n Q_n
        ok = mbar_wait_warp(qfull(s), (n / QST) & 1, abort, 38, status) &&
             mbar_wait_warp(dsfull(bb), (n / DSST) & 1, abort, 27, status);
        if (!ok) break;
        tr.ev(20);
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < C::NK_T; ++k) {
            const uint64_t bq = sdesc_sw128(sQ(s) + k * 16 * 128, C::BLK_BYTES, 1024);
            if constexpr (C::DK_TS) {
              mma_ts<MmaKind::kBF16>(tmem + C::DK_COL, tmem + C::DST_COL + 8 * k, bq, idDK,
                                     (n > 0 || k > 0) ? 1u : 0u);
            } else {
              const uint32_t off = (k / 4) * C::BLK_BYTES + (k % 4) * 32;
              mma_ss<MmaKind::kBF16>(tmem + C::DK_COL, sdesc_sw128(sDS(bb) + off, 16, 1024), bq,
                                     idDK, (n > 0 || k > 0) ? 1u : 0u);
            }
          }
          mma_commit(dsempty(bb));
          mma_commit(qempty(s));
          mma_commit(bar(C_DKDONE));
        }
        __syncwarp();
        tr.ev(21);
      }
      if (elect_one()) {
        mma_commit(bar(C_FINAL));
        mma_commit(bar(C_DRAIN3));
      }
      __syncwarp();
      mbar_wait_drain(bar(C_DRAIN3), 0, 40, status);
    }
  } else if (warp >= 4 && warp < C::DQ_WARP0) {
    // ------------------------------------------------------------ compute
    // Group grp (four warps, one per TMEM lane quadrant) owns query columns
    // q0 .. q0 + 31 of every step.  Thread = key row kr (TMEM lane).
    const int grp = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int kr = quad * 32 + lane;
    const int q0 = 32 * grp;
    const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const float c = a.scale * kLog2e;
    const float2 c2 = make_float2(c, c), ns2 = make_float2(-a.scale, -a.scale);
    (void)c;
    const uint32_t pst = trow + C::P_COL + grp * C::P_GSTRIDE;
    Tracer tr(NEA_TRACE_BASE, traced && quad == 0 && (grp == 0 || grp == C::NGRP - 1),
              grp == 0 ? 4 : 5);
    // arrive once per warp, after every lane's tensor-memory accesses
    auto warp_arrive_tc = [&](uint32_t br) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(br);
    };
    // this thread's 64 bytes of the dS'^T row: block q0 / 64, chunks from (q0 % 64) / 8
    const int dsblk = q0 / 64, dsch0 = (q0 % 64) / 8;
    bool ok = true;
    for (int n = 0; n < nsteps; ++n) {
      const int bb = n % DSST;
      const int i = i0 + n % nI;
      if (!mbar_wait_warp(bar(C_SFULL), n & 1, abort, 31, status)) {
        ok = false;
        break;
      }
      tr.ev(30);
      tc_fence_after();
      uint32_t u[32];
      tmem_ld32(trow + C::S_COL + q0, u);
      tmem_ld_wait(u);
      warp_arrive_tc(bar(C_SFREE));  // S^T_n is in registers
      tr.ev(31);
      // P^T = exp2(c S'^T) = exp(scale S^T - LSE): the row term is already in
      // S'^T (padded query rows have -1e30 there, so their P is exactly 0).
      // A key past N (zero-filled by TMA) must not take part: under the
      // causal mask it lies after every real query and is masked with the
      // diagonal; without it, it is masked here.
      const bool kdead = !a.causal && j * kTile + kr >= a.N;
      // queries q0 + x with x < lim are masked (x: column within the group)
      const int lim = kdead ? 32 : (a.causal && i == j) ? kr - q0 : 0;
      uint32_t pk[16];  // P^T row, bf16 pairs (query 2t in the low half)
      auto make_p = [&](bool masked) {
#pragma unroll
        for (int t4 = 0; t4 < 8; ++t4) {
          const float2 x0 =
              __fmul2_rn(make_float2(__uint_as_float(u[4 * t4]), __uint_as_float(u[4 * t4 + 1])), c2);
          const float2 x1 = __fmul2_rn(
              make_float2(__uint_as_float(u[4 * t4 + 2]), __uint_as_float(u[4 * t4 + 3])), c2);
          float p0 = ex2(x0.x), p1 = ex2(x0.y), p2 = ex2(x1.x), p3 = ex2(x1.y);
          if (masked) {
            const int x = 4 * t4;
            if (x < lim) p0 = 0.f;
            if (x + 1 < lim) p1 = 0.f;
            if (x + 2 < lim) p2 = 0.f;
            if (x + 3 < lim) p3 = 0.f;
          }
          pk[2 * t4] = pack_bf16(p0, p1);
          pk[2 * t4 + 1] = pack_bf16(p2, p3);
        }
      };
      if (lim > 0)
        make_p(true);
      else
        make_p(false);
      tr.ev(38);
      // P^T_n goes into this group's S^T columns, already read; S^T_n was
      // only issued after dV_{n-1} had read P^T_{n-1} there
      tr.ev(39);
      tmem_st16(pst, pk);
      tmem_st_wait();
      warp_arrive_tc(bar(C_PFULL));
      tr.ev(32);
      // dS'^T = P^T o (-scale dP'^T) = P^T o (Ds - scale dP^T), Ds = scale D
      if (!mbar_wait_warp(bar(C_DPFULL), n & 1, abort, 33, status)) {
        ok = false;
        break;
      }
      tr.ev(33);
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32(trow + C::DP_COL + q0, v);
      tmem_ld_wait(v);
      warp_arrive_tc(bar(C_DPFREE));
      tr.ev(34);
      uint32_t o[16];
#pragma unroll
      for (int t4 = 0; t4 < 8; ++t4) {
        const float2 y0 =
            __fmul2_rn(make_float2(__uint_as_float(v[4 * t4]), __uint_as_float(v[4 * t4 + 1])), ns2);
        const float2 y1 = __fmul2_rn(
            make_float2(__uint_as_float(v[4 * t4 + 2]), __uint_as_float(v[4 * t4 + 3])), ns2);
        o[2 * t4] = mul_bf16x2(pk[2 * t4], pack_bf16(y0.x, y0.y));
        o[2 * t4 + 1] = mul_bf16x2(pk[2 * t4 + 1], pack_bf16(y1.x, y1.y));
      }
      tr.ev(44);
      // buffer bb is free once dK and dQ of step n - DSST have read it
      if (n >= DSST &&
          !mbar_wait_warp(dsempty(bb), ((n / DSST) - 1) & 1, abort, 34, status)) {
        ok = false;
        break;
      }
      tr.ev(45);
      if constexpr (C::DK_TS) {
        // dS'^T_n to tensor memory for the dK MMA, once dK_{n-1} has read it
        if (n > 0 && !mbar_wait_warp(bar(C_DKDONE), (n - 1) & 1, abort, 34, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st16(trow + C::DST_COL + 16 * grp, o);
      }
      // 32 queries = 64 B of this thread's 128-B row of block dsblk, swizzled
      uint8_t* dsrow = smem + C::OFF_DS + (bb * 2 + dsblk) * C::BLK_BYTES + kr * 128;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4)
        *reinterpret_cast<uint4*>(dsrow + (((dsch0 + c4) ^ (kr & 7)) << 4)) =
            make_uint4(o[4 * c4], o[4 * c4 + 1], o[4 * c4 + 2], o[4 * c4 + 3]);
      if constexpr (C::DK_TS) {
        tmem_st_wait();
        tc_fence_before();
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(dsfull(bb));
      tr.ev(35);
    }
    // epilogue: groups 0, 1 write the two column halves of dV, groups 2, 3
    // those of dK, for this CTA's key rows
    if (ok) ok = mbar_wait_warp(bar(C_FINAL), 0, abort, 35, status);
    tr.ev(36);
    if (ok) {
      tc_fence_after();
      const bool is_dk = grp >= 2;
      const int c_lo = (grp & 1) * (D / 2);
      const bool row_ok = j * kTile + kr < a.N;  // rows past N are not stored
      const size_t row =
          (static_cast<size_t>(b) * a.Hkv + g) * a.N + static_cast<size_t>(j) * kTile + kr;
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(is_dk ? a.dK : a.dV) + row * D;
      const uint32_t col = is_dk ? C::DK_COL : C::DV_COL;
      const float sgn = is_dk ? -1.f : 1.f;  // the dK accumulator holds -dK
      // dK of rotated keys -> dK of the caller's keys (RoPE)
      const float2* rcs = (is_dk && row_ok && a.rope_cs != nullptr)
                              ? a.rope_cs + static_cast<size_t>(j * kTile + kr) * (D / 2)
                              : nullptr;
#pragma unroll
      for (int cc = c_lo; cc < c_lo + D / 2; cc += 32) {
        uint32_t w32[32];
        tmem_ld32(trow + col + cc, w32);
        tmem_ld_wait(w32);
#pragma unroll
        for (int t = 0; t < 32; ++t) w32[t] = __float_as_uint(__uint_as_float(w32[t]) * sgn);
        if (rcs != nullptr) {
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            float x0 = __uint_as_float(w32[2 * t]), x1 = __uint_as_float(w32[2 * t + 1]);
            rope_inv(x0, x1, __ldg(rcs + cc / 2 + t));
            w32[2 * t] = __float_as_uint(x0);
            w32[2 * t + 1] = __float_as_uint(x1);
          }
        }
#pragma unroll
        for (int t4 = 0; t4 < 4; ++t4) {
          uint4 wv;
          wv.x = pack_bf16(__uint_as_float(w32[8 * t4 + 0]), __uint_as_float(w32[8 * t4 + 1]));
          wv.y = pack_bf16(__uint_as_float(w32[8 * t4 + 2]), __uint_as_float(w32[8 * t4 + 3]));
          wv.z = pack_bf16(__uint_as_float(w32[8 * t4 + 4]), __uint_as_float(w32[8 * t4 + 5]));
          wv.w = pack_bf16(__uint_as_float(w32[8 * t4 + 6]), __uint_as_float(w32[8 * t4 + 7]));
          if (row_ok) *reinterpret_cast<uint4*>(dst + cc + 8 * t4) = wv;
        }
      }
    }
    tr.ev(37);
  } else if (DQ && warp >= C::DQ_WARP0) {
    // ------------------------------------------------------------ dQ drain
    // Four warps (thread = query row = TMEM lane) read dQ'_n out of tensor
    // memory 64 columns at a time, release it to the dQ issuer, and move it
    // in 128 x 32 boxes through a staging buffer into TMA reduce-adds (fp32)
    // of the accumulator.
    const int quad = warp & 3;
    const int qr = quad * 32 + lane;  // query row == TMEM lane of the dQ tile
    const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const bool lead_warp = warp == C::DQ_WARP0;  // its elected lane issues the reductions
    Tracer tr(NEA_TRACE_BASE, traced && warp == C::DQ_WARP0, 6);
    for (int n = 0; n < nsteps; ++n) {
      int h, i;
      step_hi(n, h, i);
      const int bh = b * a.H + h;
      // the whole warpgroup unwinds together: it meets at named barriers below
      if (!named_bar_and(2, 128, mbar_wait_warp(bar(C_DQFULL), n & 1, abort, 36, status)))
        break;
      tr.ev(40);
      tc_fence_after();
#pragma unroll
      for (int pr = 0; pr < D / 64; ++pr) {
        uint32_t v0[32], v1[32];
        tmem_ld32(trow + C::DQ_COL + 64 * pr, v0);
        tmem_ld32(trow + C::DQ_COL + 64 * pr + 32, v1);
        tmem_ld_wait(v0);
        reg_fence(v1);
        if (pr == D / 64 - 1) {  // dQ'_n is in registers: the next dQ MMA may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(C_DQFREE));
        }
#pragma unroll
        for (int box = 0; box < 2; ++box) {
          const uint32_t(&v)[32] = box == 0 ? v0 : v1;
          // the staging buffer is free once the previous reduction has read it
          if (lead_warp) {
            if (elect_one()) bulk_wait_read0();
            __syncwarp();
          }
          named_bar_sync(2, 128);
          uint8_t* rowp = smem + C::OFF_DQ + qr * 128;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            *reinterpret_cast<uint4*>(rowp + ((ch ^ (qr & 7)) << 4)) =
                make_uint4(v[4 * ch], v[4 * ch + 1], v[4 * ch + 2], v[4 * ch + 3]);
          fence_proxy_async();
          named_bar_sync(2, 128);
          if (lead_warp) {
            if (elect_one()) {
              tma_reduce_add_3d(&a.tmdQacc, sDQ, 64 * pr + 32 * box, i * kTile, bh);
              bulk_commit();
            }
            __syncwarp();
          }
        }
      }
      tr.ev(42);
    }
    // the staging buffer must stay until the last reductions have read it;
    // their writes complete with the grid
    if (lead_warp) {
      if (elect_one()) bulk_wait_read0();
      __syncwarp();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
#ifdef NEA_TRACE
  if (threadIdx.x == 0 && blockIdx.x < kTraceCtas) g_trace_cta[3 * blockIdx.x + 1] = global_ns();
#endif
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

cudaError_t launch_bwd_pre(const BwdArgs& a, int sms, cudaStream_t stream) {
  const int npad = (a.N + kTile - 1) / kTile * kTile;
  const long long prows = static_cast<long long>(a.B) * a.H * npad;
  const int esize = a.dtype == 0 ? 2 : 4;
  const int tpr = a.d * esize / 16;
  const long long units = prows / (static_cast<long long>(kPreThreads / tpr) * kPreRows);
  // one block per unit: more blocks than fit at once keep more loads in flight
  (void)sms;
  auto grid_for = [&](auto) { return static_cast<unsigned>(units); };
  if (a.dtype == 0 && a.d == 64)
    bwd_pre_kernel<__nv_bfloat16, 64><<<grid_for(bwd_pre_kernel<__nv_bfloat16, 64>), kPreThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(a.O), static_cast<const __nv_bfloat16*>(a.dO), a.lse,
        a.delta, a.lse2, a.dq_acc, a.fold, prows, a.N, npad, a.scale);
  else if (a.dtype == 0 && a.d == 128)
    bwd_pre_kernel<__nv_bfloat16, 128><<<grid_for(bwd_pre_kernel<__nv_bfloat16, 128>), kPreThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(a.O), static_cast<const __nv_bfloat16*>(a.dO), a.lse,
        a.delta, a.lse2, a.dq_acc, a.fold, prows, a.N, npad, a.scale);
  else if (a.dtype == 1 && a.d == 64)
    bwd_pre_kernel<float, 64><<<grid_for(bwd_pre_kernel<float, 64>), kPreThreads, 0, stream>>>(
        static_cast<const float*>(a.O), static_cast<const float*>(a.dO), a.lse, a.delta, a.lse2,
        a.dq_acc, nullptr, prows, a.N, npad, a.scale);
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

cudaError_t launch_bwd_post(const BwdArgs& a, int sms, cudaStream_t stream) {
  const long long n8 = static_cast<long long>(a.B) * a.H * a.N * a.d / 8;
  const long long per_block = static_cast<long long>(kPostThreads) * kPostVecs;
  (void)sms;
  const long long blocks = (n8 + per_block - 1) / per_block;
  bwd_post_kernel<<<static_cast<unsigned>(blocks), kPostThreads, 0, stream>>>(
      a.dq_acc, static_cast<__nv_bfloat16*>(a.dQ), n8, a.rope_cs, a.N, a.d);
  return cudaGetLastError();
}

}  // namespace nea

#ifdef NEA_TRACE
// Copies the main kernel's timeline to `host` (kTraceRoles * kTraceEvents
// values, 0 where no event was recorded) and clears it for the next launch.
extern "C" int nea_trace_read_bwd(long long* host) {
  if (cudaMemcpyFromSymbol(host, nea::g_trace_bwd, sizeof(nea::g_trace_bwd)) != cudaSuccess)
    return -1;
  static long long zeros[nea::kTraceRoles * nea::kTraceEvents] = {};
  return cudaMemcpyToSymbol(nea::g_trace_bwd, zeros, sizeof(zeros)) == cudaSuccess ? 0 : -1;
}
// Copies (start ns, end ns, SM) of the main kernel's first kTraceCtas CTAs.
extern "C" int nea_trace_read_cta(long long* host) {
  return cudaMemcpyFromSymbol(host, nea::g_trace_cta, sizeof(nea::g_trace_cta)) == cudaSuccess
             ? 0
             : -1;
}
#endif
