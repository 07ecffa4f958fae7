// nea_api.cu -- the C ABI declared in include/nea_attn.h: argument checks,
// TMA descriptor encoding, workspace carving, launches, device status word.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/nea_attn.h"
#include "nea_internal.h"

namespace nea {

// Written by kernels whose bounded waits gave up; read + cleared by
// nea_attn_check_status().  One copy per device that loaded the library.
__device__ unsigned int g_status_word = 0;

namespace {

constexpr int kMaxDevices = 64;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;
unsigned int* g_status_ptr[kMaxDevices] = {};

// Driver entry point for cuTensorMapEncodeTiled, fetched through the runtime
// so the library needs no link-time dependency on libcuda.
EncodeTiledFn encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_encode;
}

// Number of SMs of the current device (cached per device).
int sm_count() {
  static int cache[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 1;
    cache[dev] = n;
  }
  return cache[dev];
}

// Device address of g_status_word on the current device.
unsigned int* status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned int*>(p);
  }
  return g_status_ptr[dev];
}

// Encoded tensor maps, reused across calls: a map depends only on the base
// address, element type and shape, so a repeated call on the same buffers
// skips the driver's encode.  Small and least-recently-used.
struct MapKey {
  const void* base;
  long long heads;
  int dt, esize, d, N, transposed;
  bool operator==(const MapKey& o) const {
    return base == o.base && heads == o.heads && dt == o.dt && esize == o.esize && d == o.d &&
           N == o.N && transposed == o.transposed;
  }
};
constexpr int kMapCache = 64;
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  unsigned long long used;  // 0: empty
};
std::mutex g_map_mu;
MapEntry g_maps[kMapCache];
unsigned long long g_map_clock = 0;

bool map_lookup(const MapKey& k, CUtensorMap* m) {
  std::lock_guard<std::mutex> lk(g_map_mu);
  for (MapEntry& e : g_maps)
    if (e.used != 0 && e.key == k) {
      e.used = ++g_map_clock;
      *m = e.map;
      return true;
    }
  return false;
}
void map_store(const MapKey& k, const CUtensorMap& m) {
  std::lock_guard<std::mutex> lk(g_map_mu);
  MapEntry* victim = &g_maps[0];
  for (MapEntry& e : g_maps) {
    if (e.used == 0) {
      victim = &e;
      break;
    }
    if (e.used < victim->used) victim = &e;
  }
  victim->key = k;
  victim->map = m;
  victim->used = ++g_map_clock;
}

// 3-D view {d, N, heads} of a [heads][N][d] array, boxes of 128 B x 128 rows
// with 128-byte swizzle (the layout the tensor-core descriptors expect).
bool encode_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, int d, int N,
               long long heads) {
  const MapKey key{base, heads, static_cast<int>(dt), esize, d, N, 0};
  if (map_lookup(key, m)) return true;
  EncodeTiledFn enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * esize,
                           static_cast<cuuint64_t>(d) * esize * static_cast<cuuint64_t>(N)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / esize), static_cast<cuuint32_t>(kTile), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  if (enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  map_store(key, *m);
  return true;
}

// 3-D view {N, d, heads} of a transposed fp32 [heads][d][N] array: boxes of
// 32 columns (128 B) x d rows, 128-byte swizzle (K-major tf32 operands).
bool encode_3d_t(CUtensorMap* m, const void* base, int d, int N, long long heads) {
  const MapKey key{base, heads, static_cast<int>(CU_TENSOR_MAP_DATA_TYPE_FLOAT32), 4, d, N, 1};
  if (map_lookup(key, m)) return true;
  EncodeTiledFn enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(d),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(N) * 4,
                           static_cast<cuuint64_t>(N) * 4 * static_cast<cuuint64_t>(d)};
  cuuint32_t box[3] = {32, static_cast<cuuint32_t>(d), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  if (enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box,
          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  map_store(key, *m);
  return true;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape / option checks shared by every entry point.  `bwd`: the checks of
// the backward, which supports fewer fp32 shapes than the forward.
int check_common(int B, int H, int Hkv, int N, int d, float scale, int causal, int dtype,
                 bool bwd = true) {
  if (B < 1 || H < 1 || Hkv < 1 || N < 1 || d < 1) return NEA_ERR_INVALID;
  if (H % Hkv != 0) return NEA_ERR_INVALID;
  if (causal != 0 && causal != 1) return NEA_ERR_INVALID;
  if (dtype != NEA_BF16 && dtype != NEA_F32) return NEA_ERR_INVALID;
  if (!std::isfinite(scale) || !(scale > 0.f)) return NEA_ERR_INVALID;
  // Grid and TMA coordinate ranges: heads and rows as int, and at most
  // B*H*ceil(N/128) CTAs in one grid dimension.
  const long long bh = static_cast<long long>(B) * H;
  if (bh > (1LL << 24) || N > (1 << 24)) return NEA_ERR_UNSUPPORTED;
  if (bh * ((N + kTile - 1) / kTile) > 0x7fffffffLL) return NEA_ERR_UNSUPPORTED;
  // element-wise kernels (dQ cast, RoPE) launch one thread per 8..32 elements
  if (bh * N > (1LL << 40) / d) return NEA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return NEA_ERR_UNSUPPORTED;
  (void)bwd;
  if (dtype == NEA_F32 && d != 64) return NEA_ERR_UNSUPPORTED;
  return NEA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// bf16: D, -L2, fp32 dQ accumulator, row-term tiles.  fp32: D, -L2, Q^T,
// dO^T, K^T (tf32).
struct WsLayout {
  size_t delta, lse2, dqacc, fold, qt, dot, kt, total;
};
// Per-row terms and the transposed fp32 operands are padded to whole 128-row
// tiles per head (npad rows); the dQ accumulator is not.
WsLayout ws_layout(int B, int H, int Hkv, int N, int d, int dtype) {
  const size_t npad = static_cast<size_t>((N + kTile - 1) / kTile) * kTile;
  const size_t rows = static_cast<size_t>(B) * H * N;
  const size_t prows = static_cast<size_t>(B) * H * npad;
  const size_t kvprows = static_cast<size_t>(B) * Hkv * npad;
  WsLayout w;
  w.delta = 0;
  w.lse2 = align256(prows * sizeof(float));
  w.dqacc = w.fold = w.qt = w.dot = w.kt = 0;
  size_t end = w.lse2 + align256(prows * sizeof(float));
  if (dtype == NEA_BF16) {
    w.dqacc = end;
    end += align256(rows * d * sizeof(float));
    w.fold = end;  // 2 tiles x 128 rows x 8 bf16 per 128-row query tile
    end += align256(prows / kTile * 4096);
  } else {
    w.qt = end;
    w.dot = w.qt + align256(prows * d * sizeof(float));
    w.kt = w.dot + align256(prows * d * sizeof(float));
    end = w.kt + align256(kvprows * d * sizeof(float));
  }
  w.total = end;
  return w;
}

}  // namespace
}  // namespace nea

using namespace nea;

extern "C" {

int nea_version(void) { return 100; }

const char* nea_status_string(int status) {
  switch (status) {
    case NEA_OK: return "ok";
    case NEA_ERR_INVALID: return "invalid argument";
    case NEA_ERR_UNSUPPORTED: return "unsupported configuration";
    case NEA_ERR_CUDA: return "CUDA error";
    case NEA_ERR_TIMEOUT: return "a kernel wait timed out";
    case NEA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    default: return "unknown status";
  }
}

static int attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                    const float* rope_cs, int B, int H, int Hkv, int N, int d, float scale,
                    int causal, int dtype, void* stream) {
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(LSE))
    return NEA_ERR_INVALID;
  int st = check_common(B, H, Hkv, N, d, scale, causal, dtype, /*bwd=*/false);
  if (st != NEA_OK) return st;
  FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  const CUtensorMapDataType dt =
      dtype == NEA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const int es = dtype == NEA_BF16 ? 2 : 4;
  const long long bh = static_cast<long long>(B) * H, bkv = static_cast<long long>(B) * Hkv;
  if (!encode_3d(&a.tmQ, Q, dt, es, d, N, bh) || !encode_3d(&a.tmK, K, dt, es, d, N, bkv) ||
      !encode_3d(&a.tmV, V, dt, es, d, N, bkv) || !encode_3d(&a.tmO, O, dt, es, d, N, bh))
    return NEA_ERR_CUDA;
  a.lse = LSE;
  a.rope_cs = reinterpret_cast<const float2*>(rope_cs);
  a.status = status_ptr();
  if (!a.status) return NEA_ERR_CUDA;
  a.B = B; a.H = H; a.Hkv = Hkv; a.N = N; a.d = d; a.causal = causal;
  a.scale = scale; a.dtype = dtype;
  return launch_fwd(a, sm_count(), static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? NEA_OK
             : NEA_ERR_CUDA;
}

int nea_attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                 int Hkv, int N, int d, float scale, int causal, int dtype, void* stream) {
  return attn_fwd(Q, K, V, O, LSE, nullptr, B, H, Hkv, N, d, scale, causal, dtype, stream);
}

int nea_attn_fwd_rope_q(const void* Q, const void* Kr, const void* V, void* O, float* LSE,
                        const float* cos_sin, int B, int H, int Hkv, int N, int d, float scale,
                        int causal, int dtype, void* stream) {
  if (!aligned16(cos_sin)) return NEA_ERR_INVALID;
  if (dtype != NEA_BF16) return NEA_ERR_UNSUPPORTED;
  return attn_fwd(Q, Kr, V, O, LSE, cos_sin, B, H, Hkv, N, d, scale, causal, dtype, stream);
}

size_t nea_attn_bwd_workspace_bytes(int B, int H, int Hkv, int N, int d, int dtype) {
  if (check_common(B, H, Hkv, N, d, 1.0f, 1, dtype) != NEA_OK) return 0;
  return ws_layout(B, H, Hkv, N, d, dtype).total;
}

// Shared by the backward entry points: checks and fills the arguments every
// stage needs.  Pointers a stage does not use may be null (need_* = false).
static int prepare_bwd(BwdArgs* a, const void* Q, const void* K, const void* V, const void* O,
                       const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                       void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int N,
                       int d, float scale, int causal, int dtype, bool need_io, bool need_main,
                       bool need_maps) {
  if (!aligned16(dQ)) return NEA_ERR_INVALID;
  if (need_io && (!aligned16(O) || !aligned16(dO) || !aligned16(LSE))) return NEA_ERR_INVALID;
  if (need_main && (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(dO) ||
                    !aligned16(dK) || !aligned16(dV)))
    return NEA_ERR_INVALID;
  int st = check_common(B, H, Hkv, N, d, scale, causal, dtype);
  if (st != NEA_OK) return st;
  const WsLayout w = ws_layout(B, H, Hkv, N, d, dtype);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < w.total)
    return NEA_ERR_WORKSPACE;
  std::memset(a, 0, sizeof(*a));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a->delta = reinterpret_cast<float*>(ws + w.delta);
  a->lse2 = reinterpret_cast<float*>(ws + w.lse2);
  a->dq_acc = dtype == NEA_BF16 ? reinterpret_cast<float*>(ws + w.dqacc) : nullptr;
  a->fold = dtype == NEA_BF16 ? reinterpret_cast<uint16_t*>(ws + w.fold) : nullptr;
  if (dtype == NEA_F32) {
    a->qt = reinterpret_cast<float*>(ws + w.qt);
    a->dot = reinterpret_cast<float*>(ws + w.dot);
    a->kt = reinterpret_cast<float*>(ws + w.kt);
  }
  if (need_maps) {
    const CUtensorMapDataType dt =
        dtype == NEA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const int es = dtype == NEA_BF16 ? 2 : 4;
    const long long bh = static_cast<long long>(B) * H, bkv = static_cast<long long>(B) * Hkv;
    if (!encode_3d(&a->tmQ, Q, dt, es, d, N, bh) || !encode_3d(&a->tmK, K, dt, es, d, N, bkv) ||
        !encode_3d(&a->tmV, V, dt, es, d, N, bkv) || !encode_3d(&a->tmdO, dO, dt, es, d, N, bh) ||
        (dtype == NEA_BF16 &&
         !encode_3d(&a->tmdQacc, a->dq_acc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, d, N, bh)))
      return NEA_ERR_CUDA;
  }
  a->status = status_ptr();  // every stage's kernels report bounded-wait timeouts
  if (!a->status) return NEA_ERR_CUDA;
  a->Q = Q; a->K = K; a->O = O; a->dO = dO; a->lse = LSE; a->dQ = dQ; a->dK = dK; a->dV = dV;
  a->B = B; a->H = H; a->Hkv = Hkv; a->N = N; a->d = d; a->causal = causal;
  a->scale = scale; a->dtype = dtype;
  return NEA_OK;
}

// The main stage: one kernel for bf16; for fp32, the tf32 transposes of Q,
// dO and K into the workspace, then the dK/dV and dQ kernels.
static int run_main(const BwdArgs& a, cudaStream_t s) {
  if (a.dtype == NEA_BF16)
    return launch_bwd_main(a, s) == cudaSuccess ? NEA_OK : NEA_ERR_CUDA;
  const long long bh = static_cast<long long>(a.B) * a.H, bkv = static_cast<long long>(a.B) * a.Hkv;
  const int npad = (a.N + kTile - 1) / kTile * kTile;
  CUtensorMap tmQt, tmdOt, tmKt;
  if (!encode_3d_t(&tmQt, a.qt, a.d, npad, bh) || !encode_3d_t(&tmdOt, a.dot, a.d, npad, bh) ||
      !encode_3d_t(&tmKt, a.kt, a.d, npad, bkv))
    return NEA_ERR_CUDA;
  if (launch_transpose_f32(static_cast<const float*>(a.Q), a.qt, bh, a.N, s) != cudaSuccess ||
      launch_transpose_f32(static_cast<const float*>(a.dO), a.dot, bh, a.N, s) != cudaSuccess ||
      launch_transpose_f32(static_cast<const float*>(a.K), a.kt, bkv, a.N, s) != cudaSuccess)
    return NEA_ERR_CUDA;
  return launch_bwd_main_f32(a, tmQt, tmdOt, tmKt, s) == cudaSuccess ? NEA_OK : NEA_ERR_CUDA;
}

int nea_attn_bwd_preprocess(const void* O, const void* dO, const float* LSE, void* dQ,
                            void* workspace, size_t workspace_bytes, int B, int H, int Hkv,
                            int N, int d, float scale, int dtype, void* stream) {
  BwdArgs a;
  int st = prepare_bwd(&a, nullptr, nullptr, nullptr, O, dO, LSE, dQ, nullptr, nullptr, workspace,
                       workspace_bytes, B, H, Hkv, N, d, scale, 1, dtype, true, false, false);
  if (st != NEA_OK) return st;
  return launch_bwd_pre(a, sm_count(), static_cast<cudaStream_t>(stream)) == cudaSuccess ? NEA_OK
                                                                             : NEA_ERR_CUDA;
}

int nea_attn_bwd_main(const void* Q, const void* K, const void* V, const void* dO, void* dQ,
                      void* dK, void* dV, void* workspace, size_t workspace_bytes, int B, int H,
                      int Hkv, int N, int d, float scale, int causal, int dtype, void* stream) {
  BwdArgs a;
  int st = prepare_bwd(&a, Q, K, V, nullptr, dO, nullptr, dQ, dK, dV, workspace, workspace_bytes,
                       B, H, Hkv, N, d, scale, causal, dtype, false, true, true);
  if (st != NEA_OK) return st;
  return run_main(a, static_cast<cudaStream_t>(stream));
}

int nea_attn_bwd_finalize(void* dQ, void* workspace, size_t workspace_bytes, int B, int H,
                          int Hkv, int N, int d, int dtype, void* stream) {
  BwdArgs a;
  int st = prepare_bwd(&a, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, dQ, nullptr,
                       nullptr, workspace, workspace_bytes, B, H, Hkv, N, d, 1.0f, 1, dtype,
                       false, false, false);
  if (st != NEA_OK) return st;
  if (dtype != NEA_BF16) return NEA_OK;
  return launch_bwd_post(a, sm_count(), static_cast<cudaStream_t>(stream)) == cudaSuccess ? NEA_OK
                                                                              : NEA_ERR_CUDA;
}

int nea_attn_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* LSE, void* dQ, void* dK, void* dV, void* workspace,
                 size_t workspace_bytes, int B, int H, int Hkv, int N, int d, float scale,
                 int causal, int dtype, void* stream) {
  BwdArgs a;
  int st = prepare_bwd(&a, Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes, B, H, Hkv,
                       N, d, scale, causal, dtype, true, true, true);
  if (st != NEA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_bwd_pre(a, sm_count(), s) != cudaSuccess) return NEA_ERR_CUDA;
  st = run_main(a, s);
  if (st != NEA_OK) return st;
  if (dtype == NEA_BF16 && launch_bwd_post(a, sm_count(), s) != cudaSuccess) return NEA_ERR_CUDA;
  return NEA_OK;
}

int nea_rope_table(float* cos_sin, int N, int d, double base, void* stream) {
  if (!cos_sin || (reinterpret_cast<uintptr_t>(cos_sin) & 7u) != 0) return NEA_ERR_INVALID;
  if (N < 1 || N > (1 << 24) || d < 2 || d > 4096 || (d & 1) || !std::isfinite(base) ||
      !(base > 0.0))
    return NEA_ERR_INVALID;
  return launch_rope_table(reinterpret_cast<float2*>(cos_sin), N, d, base,
                           static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? NEA_OK
             : NEA_ERR_CUDA;
}

int nea_rope_qk(const void* Q, const void* K, void* Qr, void* Kr, const float* cos_sin, int B,
                int H, int Hkv, int N, int d, int dtype, void* stream) {
  if (!aligned16(Q) || !aligned16(K) || !aligned16(Qr) || !aligned16(Kr) || !aligned16(cos_sin))
    return NEA_ERR_INVALID;
  int st = check_common(B, H, Hkv, N, d, 1.0f, 1, dtype, /*bwd=*/false);
  if (st != NEA_OK) return st;
  const long long qrows = static_cast<long long>(B) * H * N;
  const long long krows = static_cast<long long>(B) * Hkv * N;
  return launch_rope_rotate(Q, K, Qr, Kr, reinterpret_cast<const float2*>(cos_sin), qrows, krows,
                            N, d, dtype, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? NEA_OK
             : NEA_ERR_CUDA;
}

int nea_attn_bwd_ex(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                    const float* LSE, const float* rope_cos_sin, int flags, void* dQ, void* dK,
                    void* dV, void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int N,
                    int d, float scale, int causal, int dtype, void* stream) {
  if ((flags & ~NEA_BWD_DETERMINISTIC) != 0) return NEA_ERR_INVALID;
  if (rope_cos_sin != nullptr && !aligned16(rope_cos_sin)) return NEA_ERR_INVALID;
  BwdArgs a;
  int st = prepare_bwd(&a, Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes, B, H,
                       Hkv, N, d, scale, causal, dtype, true, true, true);
  if (st != NEA_OK) return st;
  a.rope_cs = reinterpret_cast<const float2*>(rope_cos_sin);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == NEA_BF16 && (flags & NEA_BWD_DETERMINISTIC)) {
    // dK, dV from the main kernel without its dQ part; dQ from one CTA per
    // query tile; no accumulator to clear or cast
    a.deterministic = 1;
    a.dq_acc = nullptr;
    if (launch_bwd_pre(a, sm_count(), s) != cudaSuccess || launch_bwd_main(a, s) != cudaSuccess ||
        launch_bwd_dq(a, s) != cudaSuccess)
      return NEA_ERR_CUDA;
    return NEA_OK;
  }
  // fp32 already owns each dQ tile in one CTA, so it is deterministic as is
  if (launch_bwd_pre(a, sm_count(), s) != cudaSuccess) return NEA_ERR_CUDA;
  st = run_main(a, s);
  if (st != NEA_OK) return st;
  if (dtype == NEA_BF16 && launch_bwd_post(a, sm_count(), s) != cudaSuccess) return NEA_ERR_CUDA;
  return NEA_OK;
}

int nea_attn_bwd_rope(const void* Qr, const void* Kr, const void* V, const void* O,
                      const void* dO, const float* LSE, const float* cos_sin, void* dQ, void* dK,
                      void* dV, void* workspace, size_t workspace_bytes, int B, int H, int Hkv,
                      int N, int d, float scale, int causal, int dtype, void* stream) {
  if (!aligned16(cos_sin)) return NEA_ERR_INVALID;
  return nea_attn_bwd_ex(Qr, Kr, V, O, dO, LSE, cos_sin, 0, dQ, dK, dV, workspace,
                         workspace_bytes, B, H, Hkv, N, d, scale, causal, dtype, stream);
}

static int decode_checks(int B, int H, int Hkv, int nq, int Lmax, int d, int dtype) {
  if (B < 1 || H < 1 || Hkv < 1 || nq < 1 || Lmax < nq || H % Hkv != 0) return NEA_ERR_INVALID;
  if (dtype != NEA_BF16 && dtype != NEA_F32) return NEA_ERR_INVALID;
  if (d != 64 && d != 128) return NEA_ERR_UNSUPPORTED;
  if ((H / Hkv) * nq > kMaxDecodeRows) return NEA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hkv > 65535 || Lmax > (1 << 24) ||
      static_cast<long long>(B) * H * nq > (1LL << 30))
    return NEA_ERR_UNSUPPORTED;
  return NEA_OK;
}

size_t nea_attn_decode_workspace_bytes(int B, int H, int Hkv, int nq, int Lmax, int d) {
  if (decode_checks(B, H, Hkv, nq, Lmax, d, NEA_BF16) != NEA_OK) return 0;
  const size_t rows = static_cast<size_t>(B) * H * nq;
  const size_t nchunk = (static_cast<size_t>(Lmax) + decode_chunk_rows() - 1) / decode_chunk_rows();
  return align256(rows * nchunk * d * sizeof(float)) + align256(rows * nchunk * sizeof(float2));
}

int nea_attn_decode(const void* Q, const void* Kc, const void* Vc, const int* lens, void* O,
                    float* LSE, void* workspace, size_t workspace_bytes, int B, int H, int Hkv,
                    int nq, int Lmax, int d, float scale, int dtype, void* stream) {
  if (!aligned16(Q) || !aligned16(Kc) || !aligned16(Vc) || !aligned16(O) || !aligned16(LSE) ||
      !lens || (reinterpret_cast<uintptr_t>(lens) & 3u) != 0)
    return NEA_ERR_INVALID;
  if (!std::isfinite(scale) || !(scale > 0.f)) return NEA_ERR_INVALID;
  int st = decode_checks(B, H, Hkv, nq, Lmax, d, dtype);
  if (st != NEA_OK) return st;
  const size_t need = nea_attn_decode_workspace_bytes(B, H, Hkv, nq, Lmax, d);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < need)
    return NEA_ERR_WORKSPACE;
  DecodeArgs a;
  std::memset(&a, 0, sizeof(a));
  const size_t rows = static_cast<size_t>(B) * H * nq;
  const int chunks = (Lmax + decode_chunk_rows() - 1) / decode_chunk_rows();
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.opart = reinterpret_cast<float*>(ws);
  a.ml = reinterpret_cast<float2*>(ws + align256(rows * chunks * d * sizeof(float)));
  // the launcher splits the chunks over one wave of CTAs; the workspace holds
  // one split per chunk, the most it can choose
  a.nchunk = chunks;
  a.cps = 1;
  const long long bg = static_cast<long long>(B) * Hkv;
  const CUtensorMapDataType dt =
      dtype == NEA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const int es = dtype == NEA_BF16 ? 2 : 4;
  if (!encode_3d(&a.tmK, Kc, dt, es, d, Lmax, bg) || !encode_3d(&a.tmV, Vc, dt, es, d, Lmax, bg))
    return NEA_ERR_CUDA;
  a.Q = Q; a.Kc = Kc; a.Vc = Vc; a.lens = lens; a.O = O; a.lse = LSE;
  a.status = status_ptr();
  if (!a.status) return NEA_ERR_CUDA;
  a.B = B; a.H = H; a.Hkv = Hkv; a.nq = nq; a.Lmax = Lmax; a.d = d; a.dtype = dtype;
  a.scale = scale;
  return launch_decode(a, sm_count(), static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? NEA_OK
             : NEA_ERR_CUDA;
}

int nea_attn_check_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return NEA_ERR_CUDA;
  unsigned int word = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof(word)) != cudaSuccess) return NEA_ERR_CUDA;
  if (word != 0 && cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess)
    return NEA_ERR_CUDA;
  if (word & kStatusBadLength) return NEA_ERR_INVALID;
  return word != 0 ? NEA_ERR_TIMEOUT : NEA_OK;
}

}  // extern "C"
