// decode.cu -- attention of the newest nq tokens against a key/value cache.
//
// The pages say the model's inference works ("NanoEuler: Hand-writing GPT-2
// in Pure C/CUDA", FAQ on production inference) on a plain cache.  Reading
// taken: batch element b holds lens[b] cache rows that include the nq new
// tokens; new token t sits at position lens[b] - nq + t and sees rows up to
// it (the decoder's causal mask); query head h reads KV head h / (H / Hkv).
//
// A decode step reads the whole cache once per KV head and does a handful of
// flops per byte, so it is HBM-bound and too narrow (G * nq query rows per KV
// head) for tensor-core tiles.  Split over the cache length:
//  decode_partial  one CTA per (128-row cache chunk, batch, KV head), 128
//                  threads: scores of the group's G * nq query rows against
//                  the chunk (thread = cache row, 16-byte coalesced loads),
//                  the chunk's softmax max / sum per row, and its partial
//                  P V (thread = output column) into the workspace;
//  decode_combine  per query row, rescales the chunks' partials to the
//                  common max and normalises: O (dtype) and LSE (natural log).
// A short cache runs the first kernel alone: the splits of a (batch, KV
// head) form a thread-block cluster and fold their results on chip.
#include <algorithm>

#include <cuda_bf16.h>

#include "nea_internal.h"
#include "ptx.cuh"

namespace nea {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kChunk = 128;

__device__ __forceinline__ void unpack(const uint4& u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    v[2 * k] = __uint_as_float(w[k] << 16);
    v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
  }
}
__device__ __forceinline__ void unpack(const uint4& u, float (&v)[4]) {
  v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
  v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
}
// CPL (2 or 4) consecutive elements as fp32, in one shared-memory load.
template <int CPL>
__device__ __forceinline__ void load_cols(const __nv_bfloat16* p, float* v) {
  if constexpr (CPL == 2) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    v[0] = __uint_as_float(w << 16);
    v[1] = __uint_as_float(w & 0xffff0000u);
  } else {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    v[0] = __uint_as_float(w.x << 16);
    v[1] = __uint_as_float(w.x & 0xffff0000u);
    v[2] = __uint_as_float(w.y << 16);
    v[3] = __uint_as_float(w.y & 0xffff0000u);
  }
}
template <int CPL>
__device__ __forceinline__ void load_cols(const float* p, float* v) {
  if constexpr (CPL == 2) {
    const float2 w = *reinterpret_cast<const float2*>(p);
    v[0] = w.x; v[1] = w.y;
  } else {
    const float4 w = *reinterpret_cast<const float4*>(p);
    v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
  }
}
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ void from_f(float x, __nv_bfloat16* p) { *p = __float2bfloat16_rn(x); }
__device__ __forceinline__ void from_f(float x, float* p) { *p = x; }

// Valid cache length of batch element b; an out-of-range length is flagged
// in the status word and clamped, so that no access leaves the cache.
__device__ __forceinline__ int cache_len(const DecodeArgs& a, int b) {
  const int L = a.lens[b];
  if (L < a.nq || L > a.Lmax) {
    atomicOr(a.status, kStatusBadLength);
    return L < a.nq ? a.nq : a.Lmax;
  }
  return L;
}

// RM: the query-row bound the loops are unrolled for (the smallest of 4, 8,
// 16, 32 that holds G * nq), so that no work is spent on absent rows.
//
// One CTA per (split, batch, KV head) streams `cps` consecutive 128-row
// chunks of the cache through a ring of STAGES shared-memory stages filled
// by TMA (K and V tiles, 128-byte swizzle: a thread reading its own key row
// and a warp reading one V row both touch distinct banks); the CTAs that
// share an SM keep its loads in flight while each computes.  Per chunk:
// scores (thread = cache row), the chunk's row max and P, then P V (warp w
// owns rows w, w + 4, ...; lane l owns CPL adjacent columns) folded into a
// running (max, sum, O) per row -- the online softmax across the split.
//
// CLUSTER (a short cache): the splits of one (batch, KV head) form a thread-
// block cluster (gridDim.x = the splits = the cluster's size).  Each leaves
// its running (max, sum, O) per row in its own shared memory; after a
// cluster barrier, each rank folds one slice of the outputs over all the
// splits through distributed shared memory and writes its O and LSE
// values: one launch, no partials in global memory, no combine kernel.  A split past its element's cache, and a CTA unwinding
// after a timeout, still meet the cluster at both barriers.
template <typename T, int D, int RM, int STAGES, bool CLUSTER>
__global__ void __launch_bounds__(kChunk) decode_partial_kernel(const __grid_constant__ DecodeArgs a) {
  constexpr int ES = static_cast<int>(sizeof(T));
  constexpr int TILE = kChunk * D * ES;     // one K or V tile
  constexpr int NBLK = D * ES / 128;        // 128-byte column blocks per row
  constexpr int BLK = kChunk * 128;         // bytes per block
  constexpr int EV = 16 / ES;               // elements per 16-byte chunk
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  // K and V of a stage land on separate barriers: K is released (and the
  // stage's next K issued) once the scores have read it, while P V still
  // reads V, so that each load's latency hides under compute of the chunk
  // before the one that needs it
  __shared__ __align__(8) uint64_t fullK[STAGES], fullV[STAGES];
  __shared__ int abort_sh;
  float* q_s = reinterpret_cast<float*>(smem + 2 * STAGES * TILE);  // [RM][D], log2 units
  float* p_s = q_s + RM * D;                                        // [RM][kChunk]
  float* red = p_s + RM * kChunk;                                   // [2][4][RM]
  float* red_o = red + 8 * RM;  // RM == 4: [4 warps][4 rows][D] partial P V
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, bg = blockIdx.y;
  const int b = bg / a.Hkv, g = bg % a.Hkv, G = a.H / a.Hkv, R = G * a.nq;
  const int L = cache_len(a, b);
  const int nvc = (L + kChunk - 1) / kChunk;  // chunks holding valid rows
  const int cb = split * a.cps;
  const int ce = min(cb + a.cps, nvc);
  if (!CLUSTER && cb >= ce) return;  // past this element's cache: the combine skips the split
  const int n = ce > cb ? ce - cb : 0;
  volatile int* abort = &abort_sh;
  auto sK = [&](int s) { return smem + 2 * s * TILE; };
  auto sV = [&](int s) { return smem + (2 * s + 1) * TILE; };
  // thread 0: K (V) of chunk cb + it into stage it % STAGES
  auto issue_k = [&](int it) {
    const int s = it % STAGES;
    const uint32_t bar = smem_u32(&fullK[s]);
    mbar_expect_tx(bar, TILE);
    for (int k = 0; k < NBLK; ++k)
      tma_load_3d(smem_u32(sK(s) + k * BLK), &a.tmK, bar, k * (128 / ES), (cb + it) * kChunk, bg);
  };
  auto issue_v = [&](int it) {
    const int s = it % STAGES;
    const uint32_t bar = smem_u32(&fullV[s]);
    mbar_expect_tx(bar, TILE);
    for (int k = 0; k < NBLK; ++k)
      tma_load_3d(smem_u32(sV(s) + k * BLK), &a.tmV, bar, k * (128 / ES), (cb + it) * kChunk, bg);
  };
  if (tid == 0) {
    abort_sh = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&fullK[s]), 1);
      mbar_init(smem_u32(&fullV[s]), 1);
    }
    fence_barrier_init();
    prefetch_tmap(&a.tmK);
    prefetch_tmap(&a.tmV);
  }
  __syncthreads();
  int issued_k = 0, issued_v = 0;  // chunks whose K (V) loads thread 0 has issued
  if (tid == 0)
    for (; issued_k < STAGES && issued_k < n; ++issued_k, ++issued_v) {
      issue_k(issued_k);
      issue_v(issued_v);
    }
  // query rows r = gi * nq + t of heads g*G + gi (absent rows: zeros)
  const T* Q = static_cast<const T*>(a.Q);
  const float cq = a.scale * kLog2e;
  for (int e = tid; e < RM * D; e += kChunk) {
    const int r = e / D, k = e % D, gi = r / a.nq, t = r % a.nq;
    float x = 0.f;
    if (r < R) x = to_f(Q[((static_cast<size_t>(b) * a.H + g * G + gi) * a.nq + t) * D + k]) * cq;
    q_s[e] = x;
  }
  // P V ownership: rows warp + 4 i, columns CPL * lane .. + CPL (its place in a swizzled row)
  constexpr int RW = RM / 4;
  constexpr int CPL = D / 32;
  const int cbyte = CPL * lane * ES;
  const int vblk = cbyte / 128, vchunk = (cbyte % 128) / 16, voff = cbyte % 16;
  float2 o[RW][CPL / 2];
  float m_run[RW], l_run[RW];
#pragma unroll
  for (int i = 0; i < RW; ++i) {
    m_run[i] = -INFINITY;
    l_run[i] = 0.f;
#pragma unroll
    for (int cc = 0; cc < CPL / 2; ++cc) o[i][cc] = make_float2(0.f, 0.f);
  }
  bool ok = true;
  for (int it = 0; it < n; ++it) {
    const int s = it % STAGES;
    const int c0 = (cb + it) * kChunk;
    const int jmax = min(kChunk, L - c0);  // valid rows of this chunk
    // every thread waits itself; the CTA agrees before it goes on
    ok = __syncthreads_and(mbar_wait(smem_u32(&fullK[s]), (it / STAGES) & 1, abort, 90, a.status));
    if (!ok) break;
    // scores of cache row c0 + tid, read from its swizzled row
    const int r8 = tid & 7;
    float2 acc2[RM];
#pragma unroll
    for (int r = 0; r < RM; ++r) acc2[r] = make_float2(0.f, 0.f);
    const uint8_t* krow = sK(s) + tid * 128;
#pragma unroll
    for (int bl = 0; bl < NBLK; ++bl) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint4 u = *reinterpret_cast<const uint4*>(krow + bl * BLK + ((k ^ r8) << 4));
        float kv[EV];
        unpack(u, kv);
        const int e0 = (bl * 128 + k * 16) / ES;
#pragma unroll
        for (int r = 0; r < RM; ++r) {
          if (r < R) {
            float2 sacc = acc2[r];
#pragma unroll
            for (int k4 = 0; k4 < EV; k4 += 4) {
              const float4 qv = *reinterpret_cast<const float4*>(q_s + r * D + e0 + k4);
              sacc = __ffma2_rn(make_float2(qv.x, qv.y), make_float2(kv[k4], kv[k4 + 1]), sacc);
              sacc = __ffma2_rn(make_float2(qv.z, qv.w), make_float2(kv[k4 + 2], kv[k4 + 3]), sacc);
            }
            acc2[r] = sacc;
          }
        }
      }
    }
    const int kj = c0 + tid;
    float sc[RM];
#pragma unroll
    for (int r = 0; r < RM; ++r) {
      const int pos = L - a.nq + r % a.nq;  // this row's token position
      float sv = (r < R && tid < jmax && kj <= pos) ? acc2[r].x + acc2[r].y : -INFINITY;
      sc[r] = sv;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sv = fmaxf(sv, __shfl_xor_sync(0xffffffffu, sv, off));
      if (lane == 0) red[warp * RM + r] = sv;
    }
    __syncthreads();  // K of stage s fully read: refill it
    if (tid == 0 && issued_k < n) issue_k(issued_k++);
    ok = __syncthreads_and(mbar_wait(smem_u32(&fullV[s]), (it / STAGES) & 1, abort, 92, a.status));
    if (!ok) break;
    // rows past L may hold anything: zero their V so that P V stays finite
    // (read after the next barrier)
    if (tid >= jmax) {
      uint8_t* vrow = sV(s) + tid * 128;
#pragma unroll
      for (int bl = 0; bl < NBLK; ++bl)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          *reinterpret_cast<uint4*>(vrow + bl * BLK + (k << 4)) = make_uint4(0u, 0u, 0u, 0u);
      fence_proxy_async();  // ordered before the TMA that refills this stage
    }
#pragma unroll
    for (int r = 0; r < RM; ++r) {
      const float m = fmaxf(fmaxf(red[r], red[RM + r]), fmaxf(red[2 * RM + r], red[3 * RM + r]));
      float p = m == -INFINITY ? 0.f : exp2f(sc[r] - m);
      p_s[r * kChunk + tid] = p;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
      if (lane == 0) red[4 * RM + warp * RM + r] = p;
    }
    __syncthreads();
    // fold this chunk into the running (max, sum, O) of the warp's rows
    float2 oc[RW][CPL / 2];
#pragma unroll
    for (int i = 0; i < RW; ++i)
#pragma unroll
      for (int cc = 0; cc < CPL / 2; ++cc) oc[i][cc] = make_float2(0.f, 0.f);
    const uint8_t* vcol = sV(s) + vblk * BLK + voff;
    if constexpr (RM == 4) {
      // few rows: warp w takes keys 32w .. 32w + 31 for every row, so each V
      // element is read once; the four warps' partials meet in shared memory
      float2 ok4[4][CPL / 2];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int cc = 0; cc < CPL / 2; ++cc) ok4[r][cc] = make_float2(0.f, 0.f);
#pragma unroll 2
      for (int j = 32 * warp; j < 32 * warp + 32; j += 4) {
        float pv[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float4 x = *reinterpret_cast<const float4*>(p_s + r * kChunk + j);
          pv[r][0] = x.x; pv[r][1] = x.y; pv[r][2] = x.z; pv[r][3] = x.w;
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int row = j + jj;
          float vv[CPL];
          load_cols<CPL>(reinterpret_cast<const T*>(vcol + row * 128 + ((vchunk ^ (row & 7)) << 4)), vv);
#pragma unroll
          for (int r = 0; r < 4; ++r)
            if (r < R)
#pragma unroll
              for (int cc = 0; cc < CPL / 2; ++cc)
                ok4[r][cc] = __ffma2_rn(make_float2(pv[r][jj], pv[r][jj]),
                                        make_float2(vv[2 * cc], vv[2 * cc + 1]), ok4[r][cc]);
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int cc = 0; cc < CPL / 2; ++cc)
          *reinterpret_cast<float2*>(red_o + (warp * 4 + r) * D + CPL * lane + 2 * cc) = ok4[r][cc];
      __syncthreads();
#pragma unroll
      for (int cc = 0; cc < CPL / 2; ++cc)
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float2 x = *reinterpret_cast<const float2*>(red_o + (w * 4 + warp) * D + CPL * lane + 2 * cc);
          oc[0][cc].x += x.x;
          oc[0][cc].y += x.y;
        }
    } else if (warp < R) {
#pragma unroll 2
      for (int j = 0; j < kChunk; j += 4) {
        float pv[RW][4];
#pragma unroll
        for (int i = 0; i < RW; ++i) {
          const float4 x = *reinterpret_cast<const float4*>(p_s + (warp + 4 * i) * kChunk + j);
          pv[i][0] = x.x; pv[i][1] = x.y; pv[i][2] = x.z; pv[i][3] = x.w;
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int row = j + jj;
          float vv[CPL];
          load_cols<CPL>(reinterpret_cast<const T*>(vcol + row * 128 + ((vchunk ^ (row & 7)) << 4)), vv);
#pragma unroll
          for (int i = 0; i < RW; ++i)
#pragma unroll
            for (int cc = 0; cc < CPL / 2; ++cc)
              oc[i][cc] = __ffma2_rn(make_float2(pv[i][jj], pv[i][jj]),
                                     make_float2(vv[2 * cc], vv[2 * cc + 1]), oc[i][cc]);
        }
      }
    }
    if (warp < R) {
#pragma unroll
      for (int i = 0; i < RW; ++i) {
        const int r = warp + 4 * i;
        const float mc = fmaxf(fmaxf(red[r], red[RM + r]), fmaxf(red[2 * RM + r], red[3 * RM + r]));
        const float* ps = red + 4 * RM;
        const float lc = ps[r] + ps[RM + r] + ps[2 * RM + r] + ps[3 * RM + r];
        const float mn = fmaxf(m_run[i], mc);
        const float al = mn == -INFINITY ? 1.f : exp2f(m_run[i] - mn);
        const float be = mn == -INFINITY ? 0.f : exp2f(mc - mn);
#pragma unroll
        for (int cc = 0; cc < CPL / 2; ++cc)
          o[i][cc] = __ffma2_rn(o[i][cc], make_float2(al, al),
                                __fmul2_rn(oc[i][cc], make_float2(be, be)));
        l_run[i] = fmaf(l_run[i], al, be * lc);
        m_run[i] = mn;
      }
    }
    __syncthreads();  // V of stage s fully read: refill it
    if (tid == 0 && issued_v < n) issue_v(issued_v++);
  }
  if (!ok) {
    // unwinding: let this CTA's copies land before it exits (the last load
    // issued into each stage, K and V)
    if (tid == 0) {
      for (int it = issued_k > STAGES ? issued_k - STAGES : 0; it < issued_k; ++it)
        mbar_wait_drain(smem_u32(&fullK[it % STAGES]), (it / STAGES) & 1, 91, a.status);
      for (int it = issued_v > STAGES ? issued_v - STAGES : 0; it < issued_v; ++it)
        mbar_wait_drain(smem_u32(&fullV[it % STAGES]), (it / STAGES) & 1, 93, a.status);
    }
    if (!CLUSTER) return;
  }
  if constexpr (CLUSTER) {
    // this split's (max, sum, O) per row into the first stage (every load
    // has landed and been read), [RM][D] then [RM][2]
    __syncthreads();
    float* cl_o = reinterpret_cast<float*>(smem);
    float* cl_ml = cl_o + RM * D;
#pragma unroll
    for (int i = 0; i < RW; ++i) {
      const int r = warp + 4 * i;
      if (r < R) {
#pragma unroll
        for (int cc = 0; cc < CPL / 2; ++cc) {
          cl_o[r * D + CPL * lane + 2 * cc] = o[i][cc].x;
          cl_o[r * D + CPL * lane + 2 * cc + 1] = o[i][cc].y;
        }
        if (lane == 0) {
          cl_ml[2 * r] = m_run[i];
          cl_ml[2 * r + 1] = l_run[i];
        }
      }
    }
    cluster_sync();
    if (ok) {
      // every rank folds its own slice of the R x D outputs across the
      // splits (thread = one output element)
      const uint32_t o_base = smem_u32(cl_o), ml_base = smem_u32(cl_ml);
      const int nsp = gridDim.x;
      const int per = (R * D + nsp - 1) / nsp;
      const int e_end = min(R * D, (split + 1) * per);
      for (int e = split * per + tid; e < e_end; e += kChunk) {
        const int r = e / D, col = e % D;
        float M = -INFINITY;
        for (int q = 0; q < nsp; ++q)
          M = fmaxf(M, ld_shared_cluster_f32(mapa_shared(ml_base + 8 * r, q)));
        float lt = 0.f, ot = 0.f;
        for (int q = 0; q < nsp; ++q) {
          const float m = ld_shared_cluster_f32(mapa_shared(ml_base + 8 * r, q));
          const float w = m == -INFINITY ? 0.f : exp2f(m - M);
          lt = fmaf(w, ld_shared_cluster_f32(mapa_shared(ml_base + 8 * r + 4, q)), lt);
          ot = fmaf(w, ld_shared_cluster_f32(mapa_shared(o_base + 4 * (r * D + col), q)), ot);
        }
        const int gi = r / a.nq, t = r % a.nq;
        const size_t row = (static_cast<size_t>(b) * a.H + g * G + gi) * a.nq + t;
        from_f(ot / lt, static_cast<T*>(a.O) + row * D + col);
        if (col == 0) a.lse[row] = (M + log2f(lt)) * kLn2;
      }
    }
    cluster_sync();  // each split's shared memory stays until every rank has read it
  } else {
#pragma unroll
  for (int i = 0; i < RW; ++i) {
    const int r = warp + 4 * i;
    if (r < R) {
      const int gi = r / a.nq, t = r % a.nq;
      const size_t row = (static_cast<size_t>(b) * a.H + g * G + gi) * a.nq + t;
      float* dst = a.opart + (row * a.nchunk + split) * D + CPL * lane;
#pragma unroll
      for (int cc = 0; cc < CPL / 2; ++cc) {
        dst[2 * cc] = o[i][cc].x;
        dst[2 * cc + 1] = o[i][cc].y;
      }
      if (lane == 0) a.ml[row * a.nchunk + split] = make_float2(m_run[i], l_run[i]);
    }
  }
  }
}

// One block of kCombine threads per query row: the chunks are split over
// kCombine / D groups of D threads (thread = column), so that a long cache's
// many chunks are read in parallel; the groups meet in shared memory.
constexpr int kCombine = 256;

template <typename T, int D>
__global__ void __launch_bounds__(kCombine) decode_combine_kernel(const DecodeArgs a) {
  constexpr int NG = kCombine / D;  // chunk groups
  __shared__ float red[32];
  __shared__ float part[NG][D + 1];  // per group: weighted sums of O
  __shared__ float lpart[NG];
  const long long row = blockIdx.x;
  const int tid = threadIdx.x, col = tid % D, grp = tid / D;
  const int b = static_cast<int>(row / (static_cast<long long>(a.H) * a.nq));
  const int L = cache_len(a, b);
  const int nc = ((L + kChunk - 1) / kChunk + a.cps - 1) / a.cps;  // splits with valid rows
  const float2* ml = a.ml + row * a.nchunk;
  // common max over the chunks
  float M = -INFINITY;
  for (int c = tid; c < nc; c += kCombine) M = fmaxf(M, ml[c].x);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if ((tid & 31) == 0) red[tid >> 5] = M;
  __syncthreads();
  M = red[0];
#pragma unroll
  for (int w = 1; w < kCombine / 32; ++w) M = fmaxf(M, red[w]);
  // this group's chunks, rescaled to M
  float l = 0.f, o = 0.f;
#pragma unroll 4
  for (int c = grp; c < nc; c += NG) {
    const float2 x = ml[c];
    const float w = x.x == -INFINITY ? 0.f : exp2f(x.x - M);
    l = fmaf(w, x.y, l);
    o = fmaf(w, a.opart[(row * a.nchunk + c) * D + col], o);
  }
  part[grp][col] = o;
  if (col == 0) lpart[grp] = l;
  __syncthreads();
  if (grp == 0) {
    float ot = 0.f, lt = 0.f;
#pragma unroll
    for (int k = 0; k < NG; ++k) {
      ot += part[k][col];
      lt += lpart[k];
    }
    from_f(ot / lt, static_cast<T*>(a.O) + row * D + col);
    if (col == 0) a.lse[row] = (M + log2f(lt)) * kLn2;
  }
}

// Splits: as many CTAs as fit on the GPU at once (one wave), at most one
// per chunk; each streams its run of chunks.  `a` arrives with nchunk = the
// number of chunks (the workspace's capacity) and leaves with the split
// count and chunks per split that both kernels use.
template <typename T, int D, int RM>
cudaError_t launch_partial(DecodeArgs& a, int sms, cudaStream_t stream) {
  constexpr int TILE = kChunk * D * static_cast<int>(sizeof(T));
  // One stage: each CTA then needs the least shared memory, and more CTAs
  // per SM (whose chunks interleave) hide load latency better than deeper
  // rings do (measured on a 537 MB cache, K and V on separate barriers:
  // 148 us with one stage, 164 with two, 197 with three).
  constexpr int STAGES = 1;
  const int smem = 1024 + 2 * STAGES * TILE + (RM * D + RM * kChunk + 8 * RM) * 4 +
                   (RM == 4 ? 16 * D * 4 : 0);
  auto kp = decode_partial_kernel<T, D, RM, STAGES, false>;
  cudaError_t e = cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int per_sm = 1;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kp, kChunk, smem);
  if (e != cudaSuccess) return e;
  const long long bg = static_cast<long long>(a.B) * a.Hkv;
  const long long slots = static_cast<long long>(per_sm > 0 ? per_sm : 1) * sms;
  const int chunks = a.nchunk;
  const int nsplit = static_cast<int>(std::min<long long>(chunks, std::max<long long>(1, slots / bg)));
  a.cps = (chunks + nsplit - 1) / nsplit;
  a.nchunk = (chunks + a.cps - 1) / a.cps;
  kp<<<dim3(a.nchunk, a.B * a.Hkv), kChunk, smem, stream>>>(a);
  return cudaGetLastError();
}

// A short cache (at most kClusterChunks chunks): up to 8 splits of one
// (batch, KV head) run as a cluster and fold their results on chip.
constexpr int kClusterChunks = 16;
template <typename T, int D, int RM>
cudaError_t launch_cluster(DecodeArgs& a, cudaStream_t stream) {
  constexpr int TILE = kChunk * D * static_cast<int>(sizeof(T));
  constexpr int STAGES = 4 * TILE <= 128 * 1024 ? 2 : 1;  // (fp32 at d = 128: one)
  static_assert((RM * D + 2 * RM) * 4 <= TILE, "the split's results fit in the first stage");
  const int smem = 1024 + 2 * STAGES * TILE + (RM * D + RM * kChunk + 8 * RM) * 4 +
                   (RM == 4 ? 16 * D * 4 : 0);
  auto kp = decode_partial_kernel<T, D, RM, STAGES, true>;
  cudaError_t e = cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int chunks = a.nchunk;
  const int nsplit = std::min(chunks, 8);
  a.cps = (chunks + nsplit - 1) / nsplit;
  a.nchunk = (chunks + a.cps - 1) / a.cps;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nchunk, a.B * a.Hkv);
  cfg.blockDim = dim3(kChunk);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.nchunk;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kp, a);
}

template <typename T, int D>
cudaError_t launch_t(DecodeArgs a, int sms, cudaStream_t stream) {
  const int R = (a.H / a.Hkv) * a.nq;
  if (a.nchunk <= kClusterChunks)
    return R <= 4    ? launch_cluster<T, D, 4>(a, stream)
           : R <= 8  ? launch_cluster<T, D, 8>(a, stream)
           : R <= 16 ? launch_cluster<T, D, 16>(a, stream)
                     : launch_cluster<T, D, kMaxDecodeRows>(a, stream);
  cudaError_t e = R <= 4    ? launch_partial<T, D, 4>(a, sms, stream)
                  : R <= 8  ? launch_partial<T, D, 8>(a, sms, stream)
                  : R <= 16 ? launch_partial<T, D, 16>(a, sms, stream)
                            : launch_partial<T, D, kMaxDecodeRows>(a, sms, stream);
  if (e != cudaSuccess) return e;
  const long long rows = static_cast<long long>(a.B) * a.H * a.nq;
  decode_combine_kernel<T, D><<<static_cast<unsigned>(rows), kCombine, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

int decode_chunk_rows() { return kChunk; }

cudaError_t launch_decode(const DecodeArgs& a, int sms, cudaStream_t stream) {
  if (a.dtype == 0 && a.d == 64) return launch_t<__nv_bfloat16, 64>(a, sms, stream);
  if (a.dtype == 0 && a.d == 128) return launch_t<__nv_bfloat16, 128>(a, sms, stream);
  if (a.dtype == 1 && a.d == 64) return launch_t<float, 64>(a, sms, stream);
  if (a.dtype == 1 && a.d == 128) return launch_t<float, 128>(a, sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace nea
