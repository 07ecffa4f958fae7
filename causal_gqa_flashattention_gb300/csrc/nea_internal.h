// nea_internal.h -- launcher interface between the C-ABI translation unit
// (nea_api.cu) and the kernel translation units.  Not installed.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace nea {

// Tiles are 128 query rows x 128 key rows for every kernel.
constexpr int kTile = 128;

struct FwdArgs {
  CUtensorMap tmQ, tmK, tmV, tmO;  // 3-D maps {d, N, heads}, 128-B swizzle
  float* lse;                      // [B*H*N]
  unsigned int* status;            // device status word
  int B, H, Hkv, N, d, causal;
  float scale;                     // softmax scale
  int dtype;                       // 0 bf16, 1 fp32
  const float2* rope_cs;           // null, or RoPE (cos, sin) [N][d/2]: Q is rotated in
                                   // shared memory before its first S (bf16 only)
};

struct BwdArgs {
  CUtensorMap tmQ, tmK, tmV, tmdO;  // loads, 3-D {d, N, heads}, 128-B swizzle
  CUtensorMap tmdQacc;              // fp32 reduce target {d, N, B*H}, 128-B swizzle
  const void* Q;                    // [B,H,N,d] dtype
  const void* K;                    // [B,Hkv,N,d] dtype
  const void* O;                    // [B,H,N,d] dtype
  const void* dO;
  const float* lse;                 // [B*H*N]
  float* delta;                     // workspace: D [B*H*N]
  float* lse2;                      // workspace: -LSE * log2(e) [B*H*N]
  float* dq_acc;                    // bf16: fp32 dQ accumulator [B,H,N,d]; fp32: null
  uint16_t* fold;                   // bf16: per (head, 128-row query tile) two 128 x 8
                                    // bf16 tiles of row terms for the main kernel's MMAs
                                    // (-LSE/scale, -D as hi/mid/lo parts); fp32: null
  float* qt;                        // fp32 only: tf32-rounded Q^T  [B*H][d][N]
  float* dot;                       // fp32 only: tf32-rounded dO^T [B*H][d][N]
  float* kt;                        // fp32 only: tf32-rounded K^T  [B*Hkv][d][N]
  void* dQ;                         // output
  void* dK;
  void* dV;
  const float2* rope_cs;            // null, or RoPE (cos, sin) [N][d/2]: dQ, dK are mapped
                                    // back through the inverse rotation before they are stored
  int deterministic;                // bf16: dQ by one CTA per query tile (no reductions)
  unsigned int* status;
  int B, H, Hkv, N, d, causal;
  float scale;
  int dtype;
};

// Decode attention over a key/value cache (split over the cache length).
constexpr int kMaxDecodeRows = 32;  // G * nq query rows per KV head at most
constexpr unsigned int kStatusBadLength = 2u;  // a cache length outside [nq, Lmax]
struct DecodeArgs {
  CUtensorMap tmK, tmV;  // caches as {d, Lmax, B*Hkv}, boxes of 128 B x 128 rows, 128-B swizzle
  const void* Q;       // [B][H][nq][d] dtype
  const void* Kc;      // [B][Hkv][Lmax][d] dtype
  const void* Vc;
  const int* lens;     // [B] valid cache rows per batch element (device)
  void* O;             // [B][H][nq][d] dtype
  float* lse;          // [B][H][nq]
  float* opart;        // workspace: [B*H*nq][nchunk][d] partial P V per split
  float2* ml;          // workspace: [B*H*nq][nchunk] (max, sum) per split
  unsigned int* status;
  int B, H, Hkv, nq, Lmax, d, dtype;
  int nchunk;          // splits of the cache per (batch, KV head), one CTA each (the
                       // launcher sets it from the chunk count it receives here)
  int cps;             // 128-row chunks per split (set by the launcher)
  float scale;
};
int decode_chunk_rows();

// Each launcher validates nothing (the API layer did) and returns the
// cudaError_t of its launch(es).
// bf16: a persistent wave of min(items, sms x CTAs per SM) CTAs; tf32: one CTA per item.
cudaError_t launch_fwd(const FwdArgs& a, int sms, cudaStream_t stream);
// The HBM-bound preprocess and cast run one wave of blocks over `sms` SMs.
cudaError_t launch_bwd_pre(const BwdArgs& a, int sms, cudaStream_t stream);
cudaError_t launch_bwd_main(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_post(const BwdArgs& a, int sms, cudaStream_t stream);
// Deterministic bf16 dQ: one CTA per query tile walks its key tiles in order.
cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t stream);
// fp32 path: transposes for the workspace, then the dK/dV and dQ kernels.
cudaError_t launch_transpose_f32(const float* src, float* dst, long long heads, int N,
                                 cudaStream_t stream);
cudaError_t launch_bwd_main_f32(const BwdArgs& a, const CUtensorMap& tmQt,
                                const CUtensorMap& tmdOt, const CUtensorMap& tmKt,
                                cudaStream_t stream);
// Rotary embedding: the (cos, sin) table [N][d/2], and Qr = R(Q), Kr = R(K).
cudaError_t launch_decode(const DecodeArgs& a, int sms, cudaStream_t stream);
cudaError_t launch_rope_table(float2* cs, int N, int d, double base, cudaStream_t stream);
cudaError_t launch_rope_rotate(const void* Q, const void* K, void* Qr, void* Kr,
                               const float2* cs, long long qrows, long long krows, int N, int d,
                               int dtype, cudaStream_t stream);

}  // namespace nea
