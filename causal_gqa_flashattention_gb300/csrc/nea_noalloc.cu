// nea_noalloc.cu -- a backward entry point that needs no caller workspace.
//
// nea_attn_bwd() asks its caller for a device workspace.  Some callers cannot
// provide one: a host framework that hands a plugin only the input and
// output pointers and keeps every allocation to itself, or a latency-critical
// path where cudaMalloc (which may synchronise the whole device) is not
// allowed.  nea_attn_bwd_noalloc() serves them: its scratch lives in a
// fixed-size array in the library's own device memory, reserved on every GPU
// that loads the library for as long as the process runs.
#include <cstdint>
#include <mutex>

#include "../../include/nea_attn.h"
#include "nea_internal.h"

namespace nea {
namespace {

// The layout nea_attn_bwd_workspace_bytes() describes, each part rounded up
// to 256 bytes (padded rows: N rounded up to a multiple of 128 per head).
// 32 MiB covers, e.g., B*H*N = 98304 rows at d = 64 bf16 (27.7 MB).
constexpr size_t kScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

// Host code must not take this symbol's address as a device pointer: on the
// host it names a stand-in.  The device address comes from
// cudaGetSymbolAddress below, once per device.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_dev[kMaxDevices] = {};

// Device address of g_scratch on the current device; nullptr on failure.
void* scratch_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch_dev[dev] = p;
  }
  return g_scratch_dev[dev];
}

}  // namespace
}  // namespace nea

extern "C" size_t nea_attn_bwd_noalloc_max_bytes(void) { return nea::kScratchBytes; }

extern "C" int nea_attn_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                                    const void* dO, const float* LSE, void* dQ, void* dK,
                                    void* dV, int B, int H, int Hkv, int N, int d, float scale,
                                    int causal, int dtype, void* stream) {
  const size_t need = nea_attn_bwd_workspace_bytes(B, H, Hkv, N, d, dtype);
  if (need == 0) {
    // invalid or unsupported sizes: let the regular entry point say which
    return nea_attn_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, nullptr, 0, B, H, Hkv, N, d, scale,
                        causal, dtype, stream);
  }
  if (need > nea::kScratchBytes) return NEA_ERR_WORKSPACE;
  void* scratch = nea::scratch_ptr();
  if (!scratch) return NEA_ERR_CUDA;
  return nea_attn_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, scratch, nea::kScratchBytes, B, H, Hkv, N,
                      d, scale, causal, dtype, stream);
}
