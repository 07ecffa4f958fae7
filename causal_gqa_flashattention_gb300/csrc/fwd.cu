// fwd.cu -- causal grouped-query FlashAttention forward on tcgen05 / TMEM.
//
// "NanoEuler: Hand-writing GPT-2 in Pure C/CUDA", section "Tiled
// FlashAttention": one block per query tile, an outer loop over key/value
// tiles staged in shared memory, S = Q K^T, an online softmax update, and an
// accumulated output.  Here a work item is one (batch, head, 128-row query
// tile).  bf16 CTAs are persistent: each walks a list of items (two CTAs per
// SM at d = 64), loading the next item's Q and first K/V tiles and issuing
// its first S = Q K^T while the current item's last tile and output are
// still being finished, so that most of the load latency and the output
// store overlap other work instead of being paid in full per item.  (tf32
// has no shared memory left for a separate output buffer and runs one item
// per CTA.)  Roles:
//
//   warp 0      TMA producer: per item Q, then K_j and V_j into 2-stage
//               rings, K one tile ahead of V (K_j is released after S_j,
//               V_j after P_j V_j)
//   warp 1      MMA issuer (one thread): S = Q K_j^T (SS), O += P V_j (TS,
//               P read from tensor memory); owns the TMEM allocation
//   warps 2..5  softmax: thread = query row (TMEM lane); reads S with
//               tcgen05.ld, causal mask on the diagonal tile, online max /
//               sum in the log2 domain, writes P (bf16 or tf32) back to TMEM,
//               rescales O only when the running max grew by more than 2^8;
//               epilogue O / l -> smem -> TMA store, LSE -> global
//
// Every ring stage, barrier phase and TMEM hand-off counts tiles globally
// over the CTA's items, so the pipeline runs on across item boundaries.
//
// Tensor memory (fp32 columns, lane = query row): S [0,128), O [128,128+d),
// P [128+d, ...).  Key tiles above the causal diagonal are never loaded.
#include "nea_internal.h"
#include "ptx.cuh"
#include "trace.cuh"

namespace nea {
namespace {

constexpr int pow2_cols(int n) {
  return n <= 32 ? 32 : n <= 64 ? 64 : n <= 128 ? 128 : n <= 256 ? 256 : 512;
}

template <int D, MmaKind KIND>
struct FwdCfg {
  static constexpr int ES = KIND == MmaKind::kBF16 ? 2 : 4;  // element bytes
  static constexpr int BLK_ELEMS = 128 / ES;                 // elements per 128-B row
  static constexpr int NBLK = D * ES / 128;                  // 128-B column blocks per row
  static constexpr int BLK_BYTES = kTile * 128;              // one column block of a tile
  static constexpr int TILE_BYTES = NBLK * BLK_BYTES;
  static constexpr int KPER = 32 / ES;                       // K of one MMA instruction
  static constexpr int NK_QK = D * ES / 32;
  static constexpr int NK_PV = kTile / KPER;
  static constexpr int S_COL = 0, O_COL = 128, P_COL = 128 + D;
  static constexpr int P_COLS = KIND == MmaKind::kBF16 ? 64 : 128;
  static constexpr int TMEM_COLS = pow2_cols(P_COL + P_COLS);
  static constexpr int CTAS_PER_SM = TMEM_COLS <= 256 ? 2 : 1;
  static constexpr int STAGES = 2;
  // tf32 operands must be K-major, so for tf32 a transposer warpgroup
  // (warps 6..9) rewrites each V tile as V^T [d][keys] before O += P V^T^T.
  static constexpr bool TRANSPOSE_V = KIND == MmaKind::kTF32;
  static constexpr int THREADS = TRANSPOSE_V ? 320 : 192;
  static constexpr int VT_BYTES = TRANSPOSE_V ? TILE_BYTES : 0;
  static constexpr int VT_BLK_BYTES = D * 128;  // one 32-key column block of V^T
  static_assert(STAGES >= 2, "S_{j+1} is issued before O += P_j V_j");
  // Persistent CTAs stage O in a buffer of its own (Q's buffer takes the next
  // item's Q); tf32 stages it in Q's buffer and runs one item per CTA.
  static constexpr bool PERSIST = !TRANSPOSE_V;
  static constexpr int O_BYTES = PERSIST ? TILE_BYTES : 0;
  // Q tile, per stage: K tile, V tile (, V^T), then O.  +1 KB for alignment.
  static constexpr int SMEM_BYTES =
      1024 + TILE_BYTES * (1 + 2 * STAGES) + VT_BYTES * STAGES + O_BYTES;
};

// One work item: a query tile of one (batch, head).
struct FwdItem {
  int qt, bh, nkv;
};

// Item k of this CTA.  Items are ordered longest first (the causal diagonal
// makes query tile qt cost qt + 1 key tiles) and dealt to the CTAs in a
// zig-zag (k even: CTA c takes c of the k-th round, k odd: G-1-c), which
// evens out the total work per CTA.
__device__ __forceinline__ bool fwd_item(const FwdArgs& a, int T, int k, FwdItem& it) {
  const long long G = gridDim.x, c = blockIdx.x;
  const long long BH = static_cast<long long>(a.B) * a.H;
  const long long idx = k * G + ((k & 1) ? (G - 1 - c) : c);
  if (idx >= BH * T) return false;
  it.qt = a.causal ? static_cast<int>(T - 1 - idx / BH) : static_cast<int>(idx / BH);
  it.bh = static_cast<int>(idx % BH);
  it.nkv = a.causal ? it.qt + 1 : T;
  return true;
}

// mbarrier slots
// P and O += P V are split in two halves of the key tile (keys 0..63 and
// 64..127): PFULL1/ODONE1 and PFULL2/ODONE2, so that the first half's MMAs
// run while the softmax computes the second half.
// QEMPTY: the item's S MMAs are done, Q's buffer may take the next item's Q.
// OFREE: the epilogue has read O from TMEM, the next item's P V may overwrite it.
enum : int { B_QFULL = 0, B_SFULL, B_SFREE, B_PFULL1, B_PFULL2, B_ODONE1, B_ODONE2, B_DRAIN,
             B_QREADY, B_QEMPTY, B_OFREE, B_KFULL };
// K_FULL[s] = B_KFULL + s, V_FULL[s] = B_KFULL + ST + s, V_EMPTY[s] = B_KFULL + 2 ST + s,
// K_EMPTY[s] = B_KFULL + 5 ST + s.  K and V stages are freed separately: K_j
// once S_j is done, V_j once P_j V_j is done.

#ifdef NEA_TRACE
// Timeline of CTA 0: rows 0 producer, 1 MMA issuer, 2 first softmax warp.
__device__ long long g_trace_fwd[kTraceRoles * kTraceEvents];
#define NEA_TRACE_FWD g_trace_fwd
#else
#define NEA_TRACE_FWD nullptr
#endif

constexpr float kLog2e = 1.4426950408889634f;
// Lazy rescale: O and l keep a stale row max until the true max exceeds it
// by more than this (log2 units); P is then bounded by 2^8, exact in the end.
constexpr float kRescaleLog2 = 8.0f;

template <int D, MmaKind KIND>
__global__ void __launch_bounds__(FwdCfg<D, KIND>::THREADS, FwdCfg<D, KIND>::CTAS_PER_SM)
    fwd_kernel(const __grid_constant__ FwdArgs a) {
  using C = FwdCfg<D, KIND>;
  constexpr int ST = C::STAGES;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  // + VT_FULL[s] = B_KFULL + 3 ST + s, KREADY[s] = B_KFULL + 4 ST + s (tf32)
  __shared__ __align__(8) uint64_t bars[B_KFULL + 6 * ST];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = (a.N + kTile - 1) / kTile;  // the last tile may be partial
  FwdItem first;
  if (!fwd_item(a, T, 0, first)) return;  // (the launcher makes no such CTA)
  constexpr int kMaxItems = C::PERSIST ? 0x7fffffff : 1;  // items per CTA
  auto kv_head = [&](const FwdItem& it) {
    const int b = it.bh / a.H, h = it.bh % a.H;
    return b * a.Hkv + h / (a.H / a.Hkv);
  };

  const uint32_t sQ = smem_u32(smem);
  const uint32_t sKV = sQ + C::TILE_BYTES;  // stage s: K at +2s*TILE, V at +(2s+1)*TILE
  const uint32_t sVT = sKV + 2 * ST * C::TILE_BYTES;  // stage s: V^T at +s*VT_BYTES
  const uint32_t sO = C::PERSIST ? sVT + ST * C::VT_BYTES : sQ;  // output staging
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  volatile int* abort = &abort_sh;
  unsigned int* status = a.status;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_SFREE), 128);
    mbar_init(bar(B_PFULL1), 128);
    mbar_init(bar(B_PFULL2), 128);
    mbar_init(bar(B_ODONE1), 1);
    mbar_init(bar(B_ODONE2), 1);
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_QEMPTY), 1);
    mbar_init(bar(B_OFREE), 128);
    for (int s = 0; s < 3 * ST; ++s) mbar_init(bar(B_KFULL + s), 1);
    for (int s = 0; s < 2 * ST; ++s) mbar_init(bar(B_KFULL + 3 * ST + s), 128);
    for (int s = 0; s < ST; ++s) mbar_init(bar(B_KFULL + 5 * ST + s), 1);
    mbar_init(bar(B_QREADY), 128);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&a.tmQ);
    prefetch_tmap(&a.tmK);
    prefetch_tmap(&a.tmV);
    prefetch_tmap(&a.tmO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  const bool traced = blockIdx.x == 0 && lane == 0;
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // converged warp, warp-uniform waits; one elected lane issues the copies
    {
      Tracer tr(NEA_TRACE_FWD, traced, 0);
      // K runs one tile ahead of V: K_g is read by S_g, which is issued
      // before O += P_{g-1} V_{g-1}; V_g only by P_g V_g.  A stage of K is
      // refilled once the S that read it is done, a stage of V once its P V
      // is done.  An item's Q goes out just before its first K.
      struct Cursor {
        int k, j;
        FwdItem it;
        bool valid;
      };
      auto advance = [&](Cursor& cu) {
        if (++cu.j == cu.it.nkv) {
          ++cu.k;
          cu.j = 0;
          cu.valid = cu.k < kMaxItems && fwd_item(a, T, cu.k, cu.it);
        }
      };
      Cursor ck{0, 0, first, true}, cv{0, 0, first, true};
      int gk = 0, gv = 0, qloads = 0;  // global tile index of the next K / V load
      bool ok = true;
      // One load per pass: K_0 K_1 V_0 K_2 V_1 ...; before a K that starts a
      // new item (and so first waits for the previous item's S), the V loads
      // still owed go out, so that they do not queue behind that wait.
      while (ok && (ck.valid || cv.valid)) {
        const bool v_due =
            cv.valid && (!ck.valid || gv < gk - 1 || (gv < gk && ck.j == 0 && ck.k > 0));
        if (!v_due) {
          if (ck.j == 0) {
            // Q's buffer is free once the previous item's S MMAs are done.
            if (ck.k > 0 && !mbar_wait_warp(bar(B_QEMPTY), (ck.k - 1) & 1, abort, 15, status)) {
              ok = false;
              break;
            }
            if (elect_one()) {
              mbar_expect_tx(bar(B_QFULL), C::TILE_BYTES);
              for (int kb = 0; kb < C::NBLK; ++kb)
                tma_load_3d(sQ + kb * C::BLK_BYTES, &a.tmQ, bar(B_QFULL), kb * C::BLK_ELEMS,
                            ck.it.qt * kTile, ck.it.bh);
            }
            __syncwarp();
            qloads = ck.k + 1;
          }
          const int s = gk % ST;
          if (gk >= ST &&
              !mbar_wait_warp(bar(B_KFULL + 5 * ST + s), ((gk / ST) - 1) & 1, abort, 1, status)) {
            ok = false;
            break;
          }
          const uint32_t sK = sKV + (2 * s) * C::TILE_BYTES;
          if (elect_one()) {
            mbar_expect_tx(bar(B_KFULL + s), C::TILE_BYTES);
            for (int kb = 0; kb < C::NBLK; ++kb)
              tma_load_3d(sK + kb * C::BLK_BYTES, &a.tmK, bar(B_KFULL + s), kb * C::BLK_ELEMS,
                          ck.j * kTile, kv_head(ck.it));
          }
          __syncwarp();
          tr.ev(1);
          ++gk;
          advance(ck);
        } else {
          const int s = gv % ST;
          if (gv >= ST &&
              !mbar_wait_warp(bar(B_KFULL + 2 * ST + s), ((gv / ST) - 1) & 1, abort, 17, status)) {
            ok = false;
            break;
          }
          const uint32_t sV = sKV + (2 * s + 1) * C::TILE_BYTES;
          if (elect_one()) {
            mbar_expect_tx(bar(B_KFULL + ST + s), C::TILE_BYTES);
            for (int kb = 0; kb < C::NBLK; ++kb)
              tma_load_3d(sV + kb * C::BLK_BYTES, &a.tmV, bar(B_KFULL + ST + s),
                          kb * C::BLK_ELEMS, cv.j * kTile, kv_head(cv.it));
          }
          __syncwarp();
          tr.ev(2);
          ++gv;
          advance(cv);
        }
      }
      if (!ok) {  // let the loads already issued land before the CTA exits
        // (every earlier Q and tile was waited for by the MMA thread)
        if (qloads > 0) mbar_wait_drain(bar(B_QFULL), (qloads - 1) & 1, 2, status);
        for (int t = gk - ST > 0 ? gk - ST : 0; t < gk; ++t)
          mbar_wait_drain(bar(B_KFULL + t % ST), (t / ST) & 1, 2, status);
        for (int t = gv - ST > 0 ? gv - ST : 0; t < gv; ++t)
          mbar_wait_drain(bar(B_KFULL + ST + t % ST), (t / ST) & 1, 2, status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop (waits are warp-uniform); one
    // elected lane issues each burst of MMAs and its commits.
    {
      Tracer tr(NEA_TRACE_FWD, traced, 1);
      constexpr uint32_t idS = make_idesc<KIND>(128, 128, false, false);
      constexpr uint32_t idPV = make_idesc<KIND>(128, D, false, !C::TRANSPOSE_V);
      // Q is usable once it has landed, or once it has been rounded (tf32)
      // or rotated (RoPE) in shared memory
      const int qbar = (C::TRANSPOSE_V || a.rope_cs != nullptr) ? B_QREADY : B_QFULL;
      // S for global tile g = tile j of item `it`.  After an item's last S,
      // QEMPTY hands Q's buffer back to the producer.
      auto issue_s = [&](int g, const FwdItem& it, int j) -> bool {
        const int s = g % ST;
        const int kbar = C::TRANSPOSE_V ? B_KFULL + 4 * ST + s : B_KFULL + s;
        if (!mbar_wait_warp(bar(kbar), (g / ST) & 1, abort, 3, status)) return false;
        tr.ev(10);
        tc_fence_after();
        const uint32_t sK = sKV + (2 * s) * C::TILE_BYTES;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < C::NK_QK; ++kk) {
            const uint32_t off = ((kk * 32) / 128) * C::BLK_BYTES + (kk * 32) % 128;
            mma_ss<KIND>(tmem + C::S_COL, sdesc_sw128(sQ + off, 16, 1024),
                         sdesc_sw128(sK + off, 16, 1024), idS, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(B_SFULL));
          mma_commit(bar(B_KFULL + 5 * ST + s));  // K stage free for the producer
          if (j == it.nkv - 1) mma_commit(bar(B_QEMPTY));
        }
        __syncwarp();
        tr.ev(11);
        return true;
      };
      FwdItem cur = first;
      int k = 0, g = 0;
      bool ok = mbar_wait_warp(bar(qbar), 0, abort, 4, status) && issue_s(0, cur, 0);
      while (ok) {
        FwdItem nx;
        const bool has_next = k + 1 < kMaxItems && fwd_item(a, T, k + 1, nx);
        for (int j = 0; j < cur.nkv; ++j, ++g) {
          // S_{g+1} overwrites S once the softmax has read S_g; it is issued
          // before O += P_g V_g.  At an item's last tile, the next item's
          // first S goes first only if its Q has already landed; otherwise
          // after this tile's P V, so that the Q load does not hold it up.
          bool s_late = false;
          if (j + 1 < cur.nkv || has_next) {
            if (!mbar_wait_warp(bar(B_SFREE), g & 1, abort, 5, status)) {
              ok = false;
              break;
            }
            tr.ev(12);
            if (j + 1 < cur.nkv) {
              if (!issue_s(g + 1, cur, j + 1)) {
                ok = false;
                break;
              }
            } else if (mbar_test_warp(bar(qbar), (k + 1) & 1)) {
              if (!issue_s(g + 1, nx, 0)) {
                ok = false;
                break;
              }
            } else {
              s_late = true;
            }
          }
          // The item's first P V overwrites O: the previous epilogue must
          // have read it.
          if (j == 0 && k > 0 &&
              !mbar_wait_warp(bar(B_OFREE), (k - 1) & 1, abort, 16, status)) {
            ok = false;
            break;
          }
          const int s = g % ST;
          const int vbar = C::TRANSPOSE_V ? B_KFULL + 3 * ST + s : B_KFULL + ST + s;
          if (!mbar_wait_warp(bar(vbar), (g / ST) & 1, abort, 7, status)) {
            ok = false;
            break;
          }
          const uint32_t sV = sKV + (2 * s + 1) * C::TILE_BYTES;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            if (!mbar_wait_warp(bar(hf == 0 ? B_PFULL1 : B_PFULL2), g & 1, abort, 6, status)) {
              ok = false;
              break;
            }
            tr.ev(13 + 2 * hf);
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
              for (int kk = hf * C::NK_PV / 2; kk < (hf + 1) * C::NK_PV / 2; ++kk) {
                uint64_t bdesc;
                if constexpr (C::TRANSPOSE_V)  // V^T K-major: 32-B K-step, 4 per 128-B block
                  bdesc = sdesc_sw128(
                      sVT + s * C::VT_BYTES + (kk / 4) * C::VT_BLK_BYTES + (kk % 4) * 32, 16, 1024);
                else  // V MN-major: K-step = KPER rows of 128 B
                  bdesc = sdesc_sw128(sV + kk * C::KPER * 128, C::BLK_BYTES, 1024);
                mma_ts<KIND>(tmem + C::O_COL, tmem + C::P_COL + kk * 8, bdesc, idPV,
                             (j > 0 || kk > 0) ? 1u : 0u);
              }
              if (hf == 1) mma_commit(bar(B_KFULL + 2 * ST + s));  // V stage free for the producer
              mma_commit(bar(hf == 0 ? B_ODONE1 : B_ODONE2));
            }
            __syncwarp();
            tr.ev(14 + 2 * hf);
          }
          if (!ok) break;
          if (s_late && (!mbar_wait_warp(bar(qbar), (k + 1) & 1, abort, 4, status) ||
                         !issue_s(g + 1, nx, 0))) {
            ok = false;
            break;
          }
        }
        if (!ok || !has_next) break;
        cur = nx;
        ++k;
      }
      // Everything this warp issued must finish before TMEM is freed.
      if (elect_one()) mma_commit(bar(B_DRAIN));
      __syncwarp();
      mbar_wait_drain(bar(B_DRAIN), 0, 8, status);
    }
  } else if (warp >= 6) {
    // ------------------------------------------------------------ tf32 prep
    // (tf32 only) rounds Q (once) and each K tile to tf32 in place, and
    // writes V_j transposed (and rounded) as V^T [d][keys]: thread t = key
    // row t of V_j writes column t of V^T.
    if constexpr (C::TRANSPOSE_V) {
      const int t = threadIdx.x - 192;
      // Elementwise rounding of a whole tile: thread t owns bytes
      // [t*TILE/128, (t+1)*TILE/128); the layout does not matter.
      auto round_tile = [&](uint32_t tile) {
        uint4* p = reinterpret_cast<uint4*>(smem + (tile - sQ) + t * (C::TILE_BYTES / 128));
#pragma unroll
        for (int k = 0; k < C::TILE_BYTES / 128 / 16; ++k) {
          uint4 x = p[k];
          x.x = tf32_rna(__uint_as_float(x.x));
          x.y = tf32_rna(__uint_as_float(x.y));
          x.z = tf32_rna(__uint_as_float(x.z));
          x.w = tf32_rna(__uint_as_float(x.w));
          p[k] = x;
        }
        fence_proxy_async();
      };
      int g = 0;
      bool ok = true;
      FwdItem it;
      for (int k = 0; ok && k < kMaxItems && fwd_item(a, T, k, it); ++k) {
        if (!mbar_wait_warp(bar(B_QFULL), k & 1, abort, 13, status)) break;
        round_tile(sQ);
        mbar_arrive(bar(B_QREADY));
        for (int j = 0; j < it.nkv; ++j, ++g) {
          const int s = g % ST;
          const uint32_t ph = (g / ST) & 1;
          if (!mbar_wait_warp(bar(B_KFULL + s), ph, abort, 14, status)) {
            ok = false;
            break;
          }
          round_tile(sKV + (2 * s) * C::TILE_BYTES);
          mbar_arrive(bar(B_KFULL + 4 * ST + s));
          if (!mbar_wait_warp(bar(B_KFULL + ST + s), ph, abort, 12, status)) {
            ok = false;
            break;
          }
          const uint8_t* vrow = smem + (sKV - sQ) + (2 * s + 1) * C::TILE_BYTES + t * 128;
          uint8_t* vt =
              smem + (sVT - sQ) + s * C::VT_BYTES + (t / 32) * C::VT_BLK_BYTES + (t % 4) * 4;
          const int tchunk = (t % 32) / 4;
#pragma unroll
          for (int blk = 0; blk < C::NBLK; ++blk) {
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              const float4 x = *reinterpret_cast<const float4*>(vrow + blk * C::BLK_BYTES +
                                                               ((ch ^ (t & 7)) << 4));
              const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int c = blk * 32 + ch * 4 + e;  // column of V = row of V^T
                *reinterpret_cast<uint32_t*>(vt + c * 128 + ((tchunk ^ (c & 7)) << 4)) =
                    tf32_rna(xs[e]);
              }
            }
          }
          fence_proxy_async();
          mbar_arrive(bar(B_KFULL + 3 * ST + s));
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // row of the query tile == TMEM lane
    const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const float c = a.scale * kLog2e;
    Tracer tr(NEA_TRACE_FWD, false, 2);  // (softmax events: off, the warps are at the register limit)
    // On an abort the warps keep walking the item list without waiting, so
    // that all four take part in the same named-barrier syncs.
    bool ok = true;
    int g = 0;  // global tile index
    FwdItem it;
    for (int k = 0; k < kMaxItems && fwd_item(a, T, k, it); ++k) {
      float m_ref = -INFINITY, l = 0.f;
      if (KIND == MmaKind::kBF16 && a.rope_cs != nullptr) {
        // RoPE: rotate row r of this item's Q tile in place (pairs within a
        // 16-byte chunk of the 128-byte swizzled row; fp32 arithmetic, one
        // rounding), then hand the tile to the MMA warp (QREADY).  The next
        // item's first S then waits for this rotation.
        ok = ok && mbar_wait_warp(bar(B_QFULL), k & 1, abort, 13, status);
        const int n = it.qt * kTile + r;  // position of this query row
        if (ok && n < a.N) {
          const float4* cs4 = reinterpret_cast<const float4*>(a.rope_cs + static_cast<size_t>(n) * (D / 2));
#pragma unroll
          for (int ch = 0; ch < D / 8; ++ch) {
            uint8_t* p = smem + (ch / 8) * C::BLK_BYTES + r * 128 + (((ch % 8) ^ (r & 7)) << 4);
            uint4 w = *reinterpret_cast<const uint4*>(p);
            uint32_t* wv = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const float4 t = __ldg(cs4 + 2 * ch + h2);  // pairs 4 ch + 2 h2, + 1
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float ct = e == 0 ? t.x : t.z, st = e == 0 ? t.y : t.w;
                const uint32_t x = wv[2 * h2 + e];
                const float a0 = __uint_as_float(x << 16), b0 = __uint_as_float(x & 0xffff0000u);
                wv[2 * h2 + e] = pack_bf16(fmaf(a0, ct, -(b0 * st)), fmaf(a0, st, b0 * ct));
              }
            }
            *reinterpret_cast<uint4*>(p) = w;
          }
        }
        fence_proxy_async();
        mbar_arrive(bar(B_QREADY));
      }
      for (int j = 0; ok && j < it.nkv; ++j, ++g) {
        if (!mbar_wait_warp(bar(B_SFULL), g & 1, abort, 9, status)) {
          ok = false;
          break;
        }
        tr.ev(30);
        tc_fence_after();
        uint32_t u0[32], u1[32], u2[32], u3[32];
        tmem_ld32(trow + C::S_COL + 0, u0);
        tmem_ld32(trow + C::S_COL + 32, u1);
        tmem_ld32(trow + C::S_COL + 64, u2);
        tmem_ld32(trow + C::S_COL + 96, u3);
        tmem_ld_wait(u0);
        reg_fence(u1);
        reg_fence(u2);
        reg_fence(u3);
        tc_fence_before();
        mbar_arrive(bar(B_SFREE));
        tr.ev(31);
        float sv[128];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          sv[i] = __uint_as_float(u0[i]);
          sv[32 + i] = __uint_as_float(u1[i]);
          sv[64 + i] = __uint_as_float(u2[i]);
          sv[96 + i] = __uint_as_float(u3[i]);
        }
        // Keys past `lim` are masked: above the diagonal on the diagonal tile
        // (which also covers keys past N under the causal mask: a padded key
        // lies after every real query), and keys past N on the last tile
        // otherwise.  TMA fills rows past N with zeros.
        int lim = kTile - 1;
        if (a.causal && j == it.qt) lim = r;
        else if (!a.causal && j == T - 1) lim = a.N - 1 - j * kTile;
        if (lim < kTile - 1) {
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i > lim) sv[i] = -INFINITY;
        }
        // row max as a tree (8 independent chains), not a 128-long chain
        float mv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mv[k] = sv[k];
#pragma unroll
        for (int i = 8; i < 128; i += 8) {
#pragma unroll
          for (int k = 0; k < 8; ++k) mv[k] = fmaxf(mv[k], sv[i + k]);
        }
        const float mx = fmaxf(fmaxf(fmaxf(mv[0], mv[1]), fmaxf(mv[2], mv[3])),
                               fmaxf(fmaxf(mv[4], mv[5]), fmaxf(mv[6], mv[7])));
        const float m_new = fmaxf(m_ref, mx);
        const bool need = (m_new - m_ref) * c > kRescaleLog2;  // always true on the first tile
        float alpha = 1.f;
        if (need) {
          alpha = ex2((m_ref - m_new) * c);
          m_ref = m_new;
        }
        const float moff = -m_ref * c;
        tr.ev(32);
        // exponent arguments with packed fp32x2 FMAs; row sum in 4 packed chains
        const float2 c2 = make_float2(c, c), moff2 = make_float2(moff, moff);
        float2 rs2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
        // Two halves of the key tile.  Half h of P may be overwritten once the
        // half-h MMAs of the previous tile (of this or the previous item) are
        // done (ODONE_h); O is rescaled only after both halves of tile j-1 are
        // done and before PFULL1 releases tile j.
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          if (g > 0) {
            if (!mbar_wait_warp(bar(hf == 0 ? B_ODONE1 : B_ODONE2), (g - 1) & 1, abort, 10,
                                status)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
#pragma unroll
          for (int cc = 2 * hf; cc < 2 * hf + 2; ++cc) {
            float p[32];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 x =
                  __ffma2_rn(make_float2(sv[32 * cc + i], sv[32 * cc + i + 1]), c2, moff2);
              p[i] = ex2(x.x);
              p[i + 1] = ex2(x.y);
              rs2[(i >> 1) & 3] = __fadd2_rn(rs2[(i >> 1) & 3], make_float2(p[i], p[i + 1]));
            }
            if constexpr (KIND == MmaKind::kBF16) {
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) pk[i] = pack_bf16(p[2 * i], p[2 * i + 1]);
              tmem_st16(trow + C::P_COL + 16 * cc, pk);
            } else {
              uint32_t pk[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) pk[i] = __float_as_uint(p[i]);
              tmem_st32(trow + C::P_COL + 32 * cc, pk);
            }
          }
          if (hf == 0 && j > 0 && __any_sync(0xffffffffu, need)) {
            // O rescale: needs the half-2 MMAs of tile j-1 done as well
            if (!mbar_wait_warp(bar(B_ODONE2), (g - 1) & 1, abort, 10, status)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < D; cc += 32) {
              uint32_t o[32];
              tmem_ld32(trow + C::O_COL + cc, o);
              tmem_ld_wait(o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st32(trow + C::O_COL + cc, o);
            }
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(hf == 0 ? B_PFULL1 : B_PFULL2));
          tr.ev(33 + hf);
        }
        if (!ok) break;
        const float2 r01 = __fadd2_rn(rs2[0], rs2[1]), r23 = __fadd2_rn(rs2[2], rs2[3]);
        const float rs = (r01.x + r01.y) + (r23.x + r23.y);
        l = l * alpha + rs;
      }
      // ------------------------------------------------------------ epilogue
      tr.ev(40);
      if (ok) ok = mbar_wait_warp(bar(B_ODONE2), (g - 1) & 1, abort, 11, status);
      tr.ev(41);
      if (k > 0) {  // the previous item's store must have read the staging buffer
        if (warp == 2) {
          if (elect_one()) bulk_wait_read0();
          __syncwarp();
        }
        named_bar_sync(1, 128);
      }
      if (ok) {
        tc_fence_after();
        const float inv = 1.f / l;
        // (tf32 stages O in Q's buffer: free, as every MMA of the CTA is done)
        uint8_t* orow = smem + (sO - sQ) + r * 128;
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t o[32];
          tmem_ld32(trow + C::O_COL + cc, o);
          tmem_ld_wait(o);
          if constexpr (KIND == MmaKind::kBF16) {
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {  // 4 chunks of 8 bf16 = 16 B
              const int col = cc + 8 * q8;
              const int blk = col / C::BLK_ELEMS, chunk = (col % C::BLK_ELEMS) / 8;
              uint4 v;
              v.x = pack_bf16(__uint_as_float(o[8 * q8 + 0]) * inv, __uint_as_float(o[8 * q8 + 1]) * inv);
              v.y = pack_bf16(__uint_as_float(o[8 * q8 + 2]) * inv, __uint_as_float(o[8 * q8 + 3]) * inv);
              v.z = pack_bf16(__uint_as_float(o[8 * q8 + 4]) * inv, __uint_as_float(o[8 * q8 + 5]) * inv);
              v.w = pack_bf16(__uint_as_float(o[8 * q8 + 6]) * inv, __uint_as_float(o[8 * q8 + 7]) * inv);
              *reinterpret_cast<uint4*>(orow + blk * C::BLK_BYTES + ((chunk ^ (r & 7)) << 4)) = v;
            }
          } else {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {  // 8 chunks of 4 fp32 = 16 B
              const int col = cc + 4 * q4;
              const int blk = col / C::BLK_ELEMS, chunk = (col % C::BLK_ELEMS) / 4;
              uint4 v;
              v.x = __float_as_uint(__uint_as_float(o[4 * q4 + 0]) * inv);
              v.y = __float_as_uint(__uint_as_float(o[4 * q4 + 1]) * inv);
              v.z = __float_as_uint(__uint_as_float(o[4 * q4 + 2]) * inv);
              v.w = __float_as_uint(__uint_as_float(o[4 * q4 + 3]) * inv);
              *reinterpret_cast<uint4*>(orow + blk * C::BLK_BYTES + ((chunk ^ (r & 7)) << 4)) = v;
            }
          }
        }
        tc_fence_before();
        mbar_arrive(bar(B_OFREE));  // O is in registers: the next item may overwrite it
        if (it.qt * kTile + r < a.N)  // rows past N exist only in smem; TMA clips O
          a.lse[static_cast<size_t>(it.bh) * a.N + it.qt * kTile + r] = m_ref * a.scale + logf(l);
        fence_proxy_async();
      }
      named_bar_sync(1, 128);
      if (warp == 2) {
        if (elect_one() && !*abort) {
          for (int kb = 0; kb < C::NBLK; ++kb)
            tma_store_3d(&a.tmO, sO + kb * C::BLK_BYTES, kb * C::BLK_ELEMS, it.qt * kTile, it.bh);
          bulk_commit();
        }
        __syncwarp();
      }
    }  // items
    // the staging buffer must stay until the last store has read it; its
    // writes complete with the grid
    if (warp == 2) {
      if (elect_one()) bulk_wait_read0();
      __syncwarp();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, MmaKind KIND>
cudaError_t launch_fwd_t(const FwdArgs& a, int sms, cudaStream_t stream) {
  using C = FwdCfg<D, KIND>;
  auto kern = fwd_kernel<D, KIND>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long items = static_cast<long long>(a.B) * a.H * ((a.N + kTile - 1) / kTile);
  // persistent: one wave of CTAs (no more CTAs than items: each gets one)
  const long long slots = static_cast<long long>(sms > 0 ? sms : 1) * C::CTAS_PER_SM;
  const unsigned grid = static_cast<unsigned>(C::PERSIST && slots < items ? slots : items);
  kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, int sms, cudaStream_t stream) {
  if (a.dtype == 0 && a.d == 64) return launch_fwd_t<64, MmaKind::kBF16>(a, sms, stream);
  if (a.dtype == 0 && a.d == 128) return launch_fwd_t<128, MmaKind::kBF16>(a, sms, stream);
  if (a.dtype == 1 && a.d == 64) return launch_fwd_t<64, MmaKind::kTF32>(a, sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace nea

#ifdef NEA_TRACE
// Copies the forward kernel's timeline to `host` (kTraceRoles * kTraceEvents
// values, 0 where no event was recorded) and clears it for the next launch.
extern "C" int nea_trace_read_fwd(long long* host) {
  if (cudaMemcpyFromSymbol(host, nea::g_trace_fwd, sizeof(nea::g_trace_fwd)) != cudaSuccess)
    return -1;
  static long long zeros[nea::kTraceRoles * nea::kTraceEvents] = {};
  return cudaMemcpyToSymbol(nea::g_trace_fwd, zeros, sizeof(zeros)) == cudaSuccess ? 0 : -1;
}
#endif

