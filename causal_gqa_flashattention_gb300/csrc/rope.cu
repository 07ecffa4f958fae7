// rope.cu -- rotary position embedding of Q and K rows.
//
// The pages name RoPE among the model's techniques ("NanoEuler: Hand-writing
// GPT-2 in Pure C/CUDA", FAQ on llm.c) without a formula; this is the
// original rotary embedding: the pair (x_2i, x_2i+1) of the row at position
// n turns by n * theta_i, theta_i = base^(-2i/d).
//
//  rope_table   cs[n][i] = (cos, sin)(n * theta_i), angles in fp64, stored
//               as fp32 pairs [N][d/2];
//  rope_rotate  Qr = R(Q), Kr = R(K) in one launch: a thread rotates one
//               16-byte column chunk of one position in several heads with
//               one load of its (cos, sin) pairs (fp32 arithmetic, one
//               rounding to the dtype).
// The attention kernels then run on Qr and Kr unchanged; the backward maps
// dQr, dKr back with the transposed rotation in its own epilogues.
#include <algorithm>

#include <cuda_bf16.h>

#include "nea_internal.h"

namespace nea {
namespace {

__global__ void __launch_bounds__(256) rope_table_kernel(float2* __restrict__ cs, int N, int half,
                                                         double base) {
  const long long idx = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
  if (idx >= static_cast<long long>(N) * half) return;
  const int n = static_cast<int>(idx / half), i = static_cast<int>(idx % half);
  const double theta = pow(base, -2.0 * i / (2.0 * half));
  double s, c;
  sincos(static_cast<double>(n) * theta, &s, &c);
  cs[idx] = make_float2(static_cast<float>(c), static_cast<float>(s));
}

// 16 bytes of a row, kept as loaded (4 registers) until it is rotated:
// E elements, E / 2 pairs turned by the pairs' (cos, sin) in r.
template <typename T>
struct Chunk;
template <>
struct Chunk<__nv_bfloat16> {
  static constexpr int E = 8;
  __device__ static uint4 rotate(uint4 u, const float2* r) {
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float a = __uint_as_float(w[k] << 16), b = __uint_as_float(w[k] & 0xffff0000u);
      const __nv_bfloat162 h =
          __floats2bfloat162_rn(fmaf(a, r[k].x, -(b * r[k].y)), fmaf(a, r[k].y, b * r[k].x));
      w[k] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <>
struct Chunk<float> {
  static constexpr int E = 4;
  __device__ static uint4 rotate(uint4 u, const float2* r) {
    const float a0 = __uint_as_float(u.x), b0 = __uint_as_float(u.y);
    const float a1 = __uint_as_float(u.z), b1 = __uint_as_float(u.w);
    return make_uint4(__float_as_uint(fmaf(a0, r[0].x, -(b0 * r[0].y))),
                      __float_as_uint(fmaf(a0, r[0].y, b0 * r[0].x)),
                      __float_as_uint(fmaf(a1, r[1].x, -(b1 * r[1].y))),
                      __float_as_uint(fmaf(a1, r[1].y, b1 * r[1].x)));
  }
};

// Thread = (position n, 16-byte column chunk) x a group of kRopeHeads
// heads: the heads' chunks are all loaded before the chunk's (cos, sin)
// pairs, which serve every head, and before the first store.  Heads
// [0, h0) are rows of x0 -> y0 (Q), heads [h0, h0 + h1) rows of x1 -> y1
// (K); each head has N rows.  Chunks stay packed (4 registers each) until
// they are rotated.
#ifndef NEA_ROPE_HEADS
#define NEA_ROPE_HEADS 4
#endif
constexpr int kRopeHeads = NEA_ROPE_HEADS;

template <typename T>
__global__ void __launch_bounds__(256)
    rope_rotate_kernel(const T* __restrict__ x0, T* y0, long long h0, const T* __restrict__ x1,
                       T* y1, long long h1, const float2* __restrict__ cs, int N, int d) {
  constexpr int E = Chunk<T>::E;
  const int cpr = d / E;  // chunks per row
  const long long c = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
  if (c >= static_cast<long long>(N) * cpr) return;
  const int n = static_cast<int>(c / cpr);
  const int col = static_cast<int>(c - static_cast<long long>(n) * cpr) * E;
  // element offset of (head h, row n, chunk col) within x0/y0 or x1/y1
  auto off = [&](long long h) {
    return ((h < h0 ? h : h - h0) * N + n) * static_cast<long long>(d) + col;
  };
  for (long long hb = static_cast<long long>(blockIdx.y) * kRopeHeads; hb < h0 + h1;
       hb += static_cast<long long>(gridDim.y) * kRopeHeads) {
    uint4 v[kRopeHeads];
#pragma unroll
    for (int u = 0; u < kRopeHeads; ++u) {
      const long long h = hb + u;
      if (h < h0 + h1)
        v[u] = __ldg(reinterpret_cast<const uint4*>((h < h0 ? x0 : x1) + off(h)));
    }
    float2 r[E / 2];
    const float4* t =
        reinterpret_cast<const float4*>(cs + static_cast<size_t>(n) * (d / 2) + col / 2);
#pragma unroll
    for (int k = 0; k < E / 4; ++k) {  // two pairs per 16-byte load
      const float4 w = __ldg(t + k);
      r[2 * k] = make_float2(w.x, w.y);
      r[2 * k + 1] = make_float2(w.z, w.w);
    }
#pragma unroll
    for (int u = 0; u < kRopeHeads; ++u) {
      const long long h = hb + u;
      if (h < h0 + h1)
        *reinterpret_cast<uint4*>((h < h0 ? y0 : y1) + off(h)) = Chunk<T>::rotate(v[u], r);
    }
  }
}

}  // namespace

cudaError_t launch_rope_table(float2* cs, int N, int d, double base, cudaStream_t stream) {
  const long long n = static_cast<long long>(N) * (d / 2);
  rope_table_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(cs, N, d / 2,
                                                                                 base);
  return cudaGetLastError();
}

cudaError_t launch_rope_rotate(const void* Q, const void* K, void* Qr, void* Kr,
                               const float2* cs, long long qrows, long long krows, int N, int d,
                               int dtype, cudaStream_t stream) {
  const int E = dtype == 0 ? 8 : 4;
  const long long h0 = qrows / N, h1 = krows / N;  // heads of Q, of K
  const dim3 grid(static_cast<unsigned>((static_cast<long long>(N) * (d / E) + 255) / 256),
                  static_cast<unsigned>(std::min<long long>((h0 + h1 + kRopeHeads - 1) / kRopeHeads,
                                                            65535)));
  if (dtype == 0)
    rope_rotate_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(Q), static_cast<__nv_bfloat16*>(Qr), h0,
        static_cast<const __nv_bfloat16*>(K), static_cast<__nv_bfloat16*>(Kr), h1, cs, N, d);
  else
    rope_rotate_kernel<float><<<grid, 256, 0, stream>>>(
        static_cast<const float*>(Q), static_cast<float*>(Qr), h0, static_cast<const float*>(K),
        static_cast<float*>(Kr), h1, cs, N, d);
  return cudaGetLastError();
}

}  // namespace nea
