// swa_attn_bwd_noalloc: the backward pass for callers that cannot hand the
// library a workspace.
//
// Who needs this: code whose device memory is owned entirely by someone else
// (a host framework's caching allocator, a plugin slot with a fixed call
// signature and no workspace argument, a service that pre-reserves its whole
// memory budget at start-up) and that therefore may not call cudaMalloc, nor
// ask its host for a scratch buffer, on the call path.  swa_attn_bwd needs a
// caller-provided workspace for the per-row term Delta; this variant keeps
// Delta in a fixed-size array that is part of the library image instead.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it (kNoAllocMaxRows floats, 8 MiB) until the process exits.
// Host code cannot use the array's name as a device address; the first call
// on each device looks the address up with cudaGetSymbolAddress (with that
// device current) and caches it.  Make that first call before any stream
// capture begins.  All calls share the one array: two calls whose kernels
// overlap on the GPU (different streams, or different host threads) race on
// it and give wrong results.  Delta is fully rewritten by every call before it
// is read, so the contents left by an earlier call never leak into a result.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/swa_attn.h"
#include "swa_internal.h"

namespace {

constexpr size_t kNoAllocMaxRows = size_t(1) << 21;  // B * Hq * L limit (8 MiB of fp32)
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_delta[kNoAllocMaxRows];

std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevices] = {nullptr};

// Device address of g_noalloc_delta on the current device (looked up once).
int noalloc_scratch(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SWA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_delta) != cudaSuccess || p == nullptr) return SWA_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return SWA_OK;
}

bool is_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int swa_attn_bwd_noalloc(const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, const float* o,
                                    const float* lse, const swa_bf16* dO, float* dq, float* dk, float* dv, int B,
                                    int Hq, int Hkv, int L, int D, int window, float scale, void* stream) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return SWA_ERR_NULL_POINTER;
  if (B < 1 || Hq < 1 || Hkv < 1 || L < 1) return SWA_ERR_BAD_SHAPE;
  if (Hq % Hkv != 0) return SWA_ERR_BAD_GROUPS;
  if (D != 64 && D != 128 && D != 256 && D != 512) return SWA_ERR_BAD_HEAD_DIM;
  if (window < 0) return SWA_ERR_BAD_WINDOW;
  if (!isfinite(scale)) return SWA_ERR_BAD_SCALE;
  if (Hq > 65535 || B > 65535) return SWA_ERR_TOO_LARGE;
  if ((double)B * Hq * L > (double)kNoAllocMaxRows) return SWA_ERR_NOALLOC_LIMIT;
  if (!is_aligned16(q) || !is_aligned16(k) || !is_aligned16(v) || !is_aligned16(o) || !is_aligned16(lse) ||
      !is_aligned16(dO) || !is_aligned16(dq) || !is_aligned16(dk) || !is_aligned16(dv))
    return SWA_ERR_MISALIGNED;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return SWA_ERR_CUDA;
  if (major != 10 || minor != 3) return SWA_ERR_UNSUPPORTED_DEVICE;
  float* delta = nullptr;
  const int rc = noalloc_scratch(&delta);
  if (rc != SWA_OK) return rc;

  swa::Geom g;
  g.B = B;
  g.Hq = Hq;
  g.Hkv = Hkv;
  g.L = L;
  g.Lq = L;  // self-attention only
  g.off = 0;
  g.causal = 1;
  g.D = D;
  g.W = (window >= L) ? 0 : window;
  g.G = Hq / Hkv;
  g.scale = scale;
  g.P = 0;
  g.Rc = 0;  // no shared-prefix plan
  g.sinks = nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (swa::launch_delta(g, o, dO, delta, s) != cudaSuccess) return SWA_ERR_CUDA;
  if (swa::launch_bwd_dkdv_simt(g, q, k, v, dO, lse, delta, dk, dv, s) != cudaSuccess) return SWA_ERR_CUDA;
  if (swa::launch_bwd_dq_simt(g, q, k, v, dO, lse, delta, dq, s) != cudaSuccess) return SWA_ERR_CUDA;
  return SWA_OK;
}
