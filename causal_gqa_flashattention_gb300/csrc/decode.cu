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
#include <cuda_bf16.h>

#include "nea_internal.h"

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
// Shared memory is read through broadcasts and 16-byte vectors: the kernel
// would otherwise be bound by shared-memory instructions, not by HBM.
template <typename T, int D, int RM>
__global__ void __launch_bounds__(kChunk) decode_partial_kernel(const DecodeArgs a) {
  extern __shared__ float sm[];
  float* q_s = sm;                      // [RM][D], scaled to log2 units
  float* p_s = q_s + RM * D;            // [RM][kChunk] P of the chunk
  float* red = p_s + RM * kChunk;       // [2][4 warps][RM] partial max / sum
  T* v_s = reinterpret_cast<T*>(red + 2 * 4 * RM);  // [kChunk][D], the cache's dtype
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, bg = blockIdx.y;
  const int b = bg / a.Hkv, g = bg % a.Hkv, G = a.H / a.Hkv, R = G * a.nq;
  const int L = cache_len(a, b);
  const int c0 = c * kChunk;
  if (c0 >= L) return;  // past this element's cache: the combine skips the chunk
  const T* Q = static_cast<const T*>(a.Q);
  const T* K = static_cast<const T*>(a.Kc) + (static_cast<size_t>(b) * a.Hkv + g) * a.Lmax * D;
  const T* V = static_cast<const T*>(a.Vc) + (static_cast<size_t>(b) * a.Hkv + g) * a.Lmax * D;
  const float cq = a.scale * kLog2e;
  // this thread's cache row: its keys are loaded first, as 16-byte vectors,
  // so that they are in flight together with the V chunk's loads below
  constexpr int KV = D * static_cast<int>(sizeof(T)) / 16;  // vectors per row
  constexpr int KPRE = KV <= 16 ? KV : 16;                    // preloaded vectors
  constexpr int EV = 16 / static_cast<int>(sizeof(T));        // elements per vector
  const int kj = c0 + tid;
  uint4 kreg[KPRE];
  const uint4* krow = reinterpret_cast<const uint4*>(K + static_cast<size_t>(kj < L ? kj : c0) * D);
#pragma unroll
  for (int i = 0; i < KPRE; ++i) kreg[i] = __ldg(krow + i);
  // this chunk of V (rows past L read as zero)
  for (int e = tid; e < kChunk * KV; e += kChunk) {
    const int row = e / KV, col = (e % KV) * EV;
    uint4 u = make_uint4(0u, 0u, 0u, 0u);
    if (c0 + row < L)
      u = __ldg(reinterpret_cast<const uint4*>(V + static_cast<size_t>(c0 + row) * D + col));
    *reinterpret_cast<uint4*>(v_s + row * D + col) = u;
  }
  // query rows r = gi * nq + t of heads g*G + gi (absent rows: zeros)
  for (int e = tid; e < RM * D; e += kChunk) {
    const int r = e / D, k = e % D, gi = r / a.nq, t = r % a.nq;
    float x = 0.f;
    if (r < R) x = to_f(Q[((static_cast<size_t>(b) * a.H + g * G + gi) * a.nq + t) * D + k]) * cq;
    q_s[e] = x;
  }
  __syncthreads();
  // scores of this thread's cache row against the RM rows: packed fp32
  // FMAs over element pairs, the two halves summed at the end
  float2 acc2[RM];
#pragma unroll
  for (int r = 0; r < RM; ++r) acc2[r] = make_float2(0.f, 0.f);
#pragma unroll
  for (int part = 0; part < KV / KPRE; ++part) {
    if (part > 0) {
#pragma unroll
      for (int i = 0; i < KPRE; ++i) kreg[i] = __ldg(krow + part * KPRE + i);
    }
#pragma unroll
    for (int i = 0; i < KPRE; ++i) {
      float kv[EV];
      unpack(kreg[i], kv);
      const int k0 = (part * KPRE + i) * EV;
#pragma unroll
      for (int r = 0; r < RM; ++r) {
        if (r < R) {
          float2 s = acc2[r];
#pragma unroll
          for (int k4 = 0; k4 < EV; k4 += 4) {
            const float4 qv = *reinterpret_cast<const float4*>(q_s + r * D + k0 + k4);
            s = __ffma2_rn(make_float2(qv.x, qv.y), make_float2(kv[k4], kv[k4 + 1]), s);
            s = __ffma2_rn(make_float2(qv.z, qv.w), make_float2(kv[k4 + 2], kv[k4 + 3]), s);
          }
          acc2[r] = s;
        }
      }
    }
  }
  float acc[RM];
#pragma unroll
  for (int r = 0; r < RM; ++r) acc[r] = acc2[r].x + acc2[r].y;
  // masked scores; the chunk's max per row (warp shuffles, then across warps)
#pragma unroll
  for (int r = 0; r < RM; ++r) {
    const int pos = L - a.nq + r % a.nq;  // this row's token position
    float sv = (r < R && kj < L && kj <= pos) ? acc[r] : -INFINITY;
    acc[r] = sv;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sv = fmaxf(sv, __shfl_xor_sync(0xffffffffu, sv, off));
    if (lane == 0) red[warp * RM + r] = sv;
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < RM; ++r) {
    const float m = fmaxf(fmaxf(red[r], red[RM + r]), fmaxf(red[2 * RM + r], red[3 * RM + r]));
    float p = m == -INFINITY ? 0.f : exp2f(acc[r] - m);
    p_s[r * kChunk + tid] = p;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
    if (lane == 0) red[4 * RM + warp * RM + r] = p;
    acc[r] = m;
  }
  __syncthreads();
  // partial O = P V: warp w takes rows w, w + 4, ...; lane l the CPL columns
  // from CPL * l, over all kChunk rows of the chunk
  constexpr int RW = RM / 4;   // rows per warp
  constexpr int CPL = D / 32;  // columns per lane
  float2 o[RW][CPL / 2];
#pragma unroll
  for (int i = 0; i < RW; ++i)
#pragma unroll
    for (int cc = 0; cc < CPL / 2; ++cc) o[i][cc] = make_float2(0.f, 0.f);
  const bool any = warp < R;  // this warp owns at least one present row
  if (any) {
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
        float vv[CPL];
        load_cols<CPL>(v_s + (j + jj) * D + CPL * lane, vv);
#pragma unroll
        for (int i = 0; i < RW; ++i)
#pragma unroll
          for (int cc = 0; cc < CPL / 2; ++cc)
            o[i][cc] = __ffma2_rn(make_float2(pv[i][jj], pv[i][jj]),
                                  make_float2(vv[2 * cc], vv[2 * cc + 1]), o[i][cc]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < RW; ++i) {
    const int r = warp + 4 * i;
    if (r < R) {
      const int gi = r / a.nq, t = r % a.nq;
      const size_t row = (static_cast<size_t>(b) * a.H + g * G + gi) * a.nq + t;
      float* dst = a.opart + (row * a.nchunk + c) * D + CPL * lane;
#pragma unroll
      for (int cc = 0; cc < CPL / 2; ++cc) {
        dst[2 * cc] = o[i][cc].x;
        dst[2 * cc + 1] = o[i][cc].y;
      }
      if (lane == 0) {
        const float* ps = red + 4 * RM;
        const float l = ps[r] + ps[RM + r] + ps[2 * RM + r] + ps[3 * RM + r];
        const float m = fmaxf(fmaxf(red[r], red[RM + r]), fmaxf(red[2 * RM + r], red[3 * RM + r]));
        a.ml[row * a.nchunk + c] = make_float2(m, l);
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
  const int nc = (L + kChunk - 1) / kChunk;
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

template <typename T, int D, int RM>
cudaError_t launch_partial(const DecodeArgs& a, cudaStream_t stream) {
  const int smem = (RM * D + RM * kChunk + 8 * RM) * 4 + kChunk * D * static_cast<int>(sizeof(T));
  auto kp = decode_partial_kernel<T, D, RM>;
  cudaError_t e = cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kp<<<dim3(a.nchunk, a.B * a.Hkv), kChunk, smem, stream>>>(a);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t stream) {
  const int R = (a.H / a.Hkv) * a.nq;
  cudaError_t e = R <= 4    ? launch_partial<T, D, 4>(a, stream)
                  : R <= 8  ? launch_partial<T, D, 8>(a, stream)
                  : R <= 16 ? launch_partial<T, D, 16>(a, stream)
                            : launch_partial<T, D, kMaxDecodeRows>(a, stream);
  if (e != cudaSuccess) return e;
  const long long rows = static_cast<long long>(a.B) * a.H * a.nq;
  decode_combine_kernel<T, D><<<static_cast<unsigned>(rows), kCombine, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

int decode_chunk_rows() { return kChunk; }

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.dtype == 0 && a.d == 64) return launch_t<__nv_bfloat16, 64>(a, stream);
  if (a.dtype == 0 && a.d == 128) return launch_t<__nv_bfloat16, 128>(a, stream);
  if (a.dtype == 1 && a.d == 64) return launch_t<float, 64>(a, stream);
  if (a.dtype == 1 && a.d == 128) return launch_t<float, 128>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace nea
