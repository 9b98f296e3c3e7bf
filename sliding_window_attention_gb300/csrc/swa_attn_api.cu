// C-ABI entry points: argument validation, workspace layout, the per-device
// status word, and launch orchestration on the caller's stream.  Every step
// of the computation runs in the kernels; this file only checks arguments
// and enqueues launches.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <string>
#include <vector>

#include "../../include/swa_attn.h"
#include "swa_internal.h"

namespace {

// ---- optional per-launch event timing (swa_attn_profile_begin/end) ----
struct ProfRec {
  std::string name;
  cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof_recs;

// Runs `f` (which enqueues one kernel on `s`); brackets it with events when
// profiling is on.
template <typename F>
cudaError_t launch(const char* name, cudaStream_t s, F&& f) {
  bool on;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    on = g_prof_on;
  }
  if (!on) return f();
  ProfRec r{name, nullptr, nullptr};
  if (cudaEventCreate(&r.start) != cudaSuccess || cudaEventCreate(&r.stop) != cudaSuccess) return cudaErrorUnknown;
  cudaEventRecord(r.start, s);
  const cudaError_t e = f();
  cudaEventRecord(r.stop, s);
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_recs.push_back(r);
  return e;
}

// Runs f1 then f2 (each enqueues one kernel on `s`, the second allowed to
// start before the first has finished); with profiling on, both records span
// the two launches, since an event between them would serialise them.
template <typename F1, typename F2>
cudaError_t launch_overlapped(const char* name1, const char* name2, cudaStream_t s, F1&& f1, F2&& f2) {
  bool on;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    on = g_prof_on;
  }
  if (!on) {
    const cudaError_t e = f1();
    return e != cudaSuccess ? e : f2();
  }
  ProfRec r1{name1, nullptr, nullptr}, r2{name2, nullptr, nullptr};
  if (cudaEventCreate(&r1.start) != cudaSuccess || cudaEventCreate(&r1.stop) != cudaSuccess ||
      cudaEventCreate(&r2.start) != cudaSuccess || cudaEventCreate(&r2.stop) != cudaSuccess)
    return cudaErrorUnknown;
  cudaEventRecord(r1.start, s);
  cudaEventRecord(r2.start, s);
  cudaError_t e = f1();
  if (e == cudaSuccess) e = f2();
  cudaEventRecord(r1.stop, s);
  cudaEventRecord(r2.stop, s);
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_recs.push_back(r1);
  g_prof_recs.push_back(r2);
  return e;
}

constexpr int kMaxDevices = 64;

// Per-device status word: kernels latch the first device-side error here.
__device__ int g_status_word;

int* status_ptr_for_current_device(int* err) {
  static int* cached[kMaxDevices] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = SWA_ERR_CUDA;
    return nullptr;
  }
  if (!cached[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
      *err = SWA_ERR_CUDA;
      return nullptr;
    }
    cached[dev] = static_cast<int*>(p);
  }
  *err = SWA_OK;
  return cached[dev];
}

int check_device() {
  static int ok_cache[kMaxDevices] = {0};  // 0 unknown, 1 ok, -1 bad
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SWA_ERR_CUDA;
  if (ok_cache[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return SWA_ERR_CUDA;
    ok_cache[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  return ok_cache[dev] == 1 ? SWA_OK : SWA_ERR_UNSUPPORTED_DEVICE;
}

// Whether the device can hold the cluster kernels' per-SM tile scratch
// (head dim 512 forward and backward, head dim 256 backward; checked once per
// device and kernel family).
enum ScratchUser { kScratchFwd512 = 0, kScratchBwd512 = 1, kScratchBwd256 = 2 };
int check_scratch_layout(int user) {
  static int cache[3][kMaxDevices] = {};  // 0 unknown, 1 ok, 2 unsupported
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SWA_ERR_CUDA;
  int& c = cache[user][dev];
  if (c == 0) {
    const int r = user == kScratchFwd512   ? swa::scratch_layout_fwd512()
                  : user == kScratchBwd512 ? swa::scratch_layout_bwd512()
                                           : swa::scratch_layout_bwd256();
    if (r < 0) return SWA_ERR_CUDA;
    c = r == 0 ? 1 : 2;
  }
  return c == 1 ? SWA_OK : SWA_ERR_SCRATCH_LAYOUT;
}

// Per-device side stream for the dK/dV pass of the backward, with the two
// events that fork it from and join it back to the caller's stream.  The
// dK/dV and dQ passes read the same inputs and write disjoint outputs; run
// side by side, the dQ pass takes the SMs that the dK/dV pass leaves idle
// (its last wave of one-SM CTAs at head dim 64-256; the 22 SMs outside its
// 10-CTA clusters at head dim 512).  The side
// stream has the highest priority, so a dK/dV cluster is placed first
// whenever SMs free up.  `mu` serialises the record/wait sequence, so that
// host threads sharing the events cannot interleave their forks.
struct SideStream {
  std::mutex mu;
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
SideStream g_side[kMaxDevices];

SideStream* side_stream_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  SideStream& ss = g_side[dev];
  std::lock_guard<std::mutex> lk(ss.mu);
  if (!ss.stream) {
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return nullptr;
    cudaStream_t st = nullptr;
    cudaEvent_t f = nullptr, j = nullptr;
    if (cudaStreamCreateWithPriority(&st, cudaStreamNonBlocking, greatest) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&f, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&j, cudaEventDisableTiming) != cudaSuccess) {
      if (f) cudaEventDestroy(f);
      cudaStreamDestroy(st);
      return nullptr;
    }
    ss.fork = f;
    ss.join = j;
    ss.stream = st;
  }
  return &ss;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int check_shape(int B, int Hq, int Hkv, int Lq, int L, int D, int window, float scale) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Lq < 1 || L < Lq) return SWA_ERR_BAD_SHAPE;
  if (Hq % Hkv != 0) return SWA_ERR_BAD_GROUPS;
  if (D != 64 && D != 128 && D != 256 && D != 512) return SWA_ERR_BAD_HEAD_DIM;
  if (window < 0) return SWA_ERR_BAD_WINDOW;
  if (!isfinite(scale)) return SWA_ERR_BAD_SCALE;
  // grid.y / grid.z carry heads and batch; element offsets must fit in int64 comfortably
  if (Hq > 65535 || B > 65535) return SWA_ERR_TOO_LARGE;
  const double elems = (double)B * Hq * L * D;
  if (elems > 9.0e15) return SWA_ERR_TOO_LARGE;
  return SWA_OK;
}

// L = key rows, Lq = query rows (the last Lq key positions)
swa::Geom make_geom(int B, int Hq, int Hkv, int Lq, int L, int D, int window, int causal, float scale) {
  swa::Geom g;
  g.B = B;
  g.Hq = Hq;
  g.Hkv = Hkv;
  g.L = L;
  g.Lq = Lq;
  g.off = L - Lq;
  g.D = D;
  // |a - j| <= L - 1 for every query position a and key j, so a window of L
  // or more masks nothing beyond the causal rule (or nothing at all)
  g.W = (window >= L) ? 0 : window;
  g.causal = causal ? 1 : 0;
  g.G = Hq / Hkv;
  g.scale = scale;
  g.P = 0;
  g.Rc = 0;
  g.sinks = nullptr;
  return g;
}

// A shared-prefix plan over L rows (prompt P, chosen response Rc, rejected
// response L - P - Rc): 0 for a valid plan, SWA_ERR_BAD_PLAN otherwise.
int check_plan(int L, int P, int Rc) {
  if (P < 0 || Rc < 0 || (long long)P + Rc > L) return SWA_ERR_BAD_PLAN;
  return SWA_OK;
}

// The geometry of a plan; a plan without a chosen or without a rejected
// response is the plain causal window (Rc = 0).
swa::Geom make_plan_geom(int B, int Hq, int Hkv, int L, int D, int window, int P, int Rc, float scale) {
  swa::Geom g = make_geom(B, Hq, Hkv, L, L, D, window, 1, scale);
  if (Rc > 0 && P + Rc < L) {
    g.P = P;
    g.Rc = Rc;
  }
  return g;
}

// Backward workspace layout: [Delta: B*Hq*L fp32].
size_t bwd_delta_bytes(int B, int Hq, int L) { return round_up((size_t)B * Hq * L * sizeof(float), 256); }

// Backward workspace layout on the tensor-core path:
// [row stats: lse*log2e plane, Delta plane, B*Hq*Lpad floats each; the dO
// scale tail][q16][k16][v16][dO16].
struct BwdTcWs {
  size_t stats, q16, k16, v16, g16, total;
  int Lpad;
};
BwdTcWs bwd_tc_ws_layout(int B, int Hq, int Hkv, int Lq, int L, int D) {
  BwdTcWs w;
  w.Lpad = swa::bwd_stats_lpad(Lq);
  w.stats = 0;
  w.q16 = round_up((size_t)B * Hq * w.Lpad * 8 + (size_t)swa::kDScaleTailFloats * 4, 256);
  w.k16 = w.q16 + round_up((size_t)B * Hq * Lq * D * 2, 256);
  w.v16 = w.k16 + round_up((size_t)B * Hkv * L * D * 2, 256);
  w.g16 = w.v16 + round_up((size_t)B * Hkv * L * D * 2, 256);
  w.total = w.g16 + round_up((size_t)B * Hq * Lq * D * 2, 256);
  return w;
}

// Forward workspace layout on the tensor-core path: an fp16 copy of v (S =
// Q K^T reads the bf16 q and k directly; O += P V pairs v with fp16 P), then
// the work counter of the persistent head-dim-512 forward (zeroed by the
// conversion of v, which runs first).
struct FwdWs {
  size_t v16, work, total;
};
FwdWs fwd_ws_layout(int B, int Hq, int Hkv, int Lq, int L, int D) {
  (void)Hq;
  (void)Lq;
  FwdWs w;
  w.v16 = 0;
  w.work = w.v16 + round_up((size_t)B * Hkv * L * D * 2, 256);
  w.total = w.work + 256;
  return w;
}

}  // namespace

// Workspace bytes of the forward on geometry g (the decode kernel serves at
// most 16 query rows per kv head, without a shared-prefix plan).
static size_t fwd_need(const swa::Geom& g) {
  if (swa::decode_supported(g)) return round_up(swa::decode_workspace_bytes(g), 256);
  return fwd_ws_layout(g.B, g.Hq, g.Hkv, g.Lq, g.L, g.D).total;
}

// The forward on a shape-checked geometry (the tail of swa_attn_fwd_ex and
// swa_attn_fwd_prefix).
static int fwd_run(const swa::Geom& g, const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, float* o,
                   float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  const int B = g.B, Hq = g.Hq, Hkv = g.Hkv, Lq = g.Lq, Lk = g.L, D = g.D;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 16) ||
      !aligned(workspace, 256))
    return SWA_ERR_MISALIGNED;
  const size_t need = fwd_need(g);
  if (workspace_bytes < need || (need > 0 && !workspace)) return SWA_ERR_WORKSPACE;
  int rc = check_device();
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = status_ptr_for_current_device(&rc);
  if (!status) return rc;
  if (swa::decode_supported(g)) {
    // at most 16 query rows per kv head (a decode step): one pass over the
    // bf16 cache, no fp16 copies
    float* ws = static_cast<float*>(workspace);
    if (launch("fwd_decode", s, [&] { return swa::launch_fwd_decode(g, q, k, v, o, lse, ws, status, s); }) !=
        cudaSuccess)
      return SWA_ERR_CUDA;
    return SWA_OK;
  }
  if (D == 512 && (rc = check_scratch_layout(kScratchFwd512)) != SWA_OK) return rc;
  const FwdWs w = fwd_ws_layout(B, Hq, Hkv, Lq, Lk, D);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  uint16_t* v16 = reinterpret_cast<uint16_t*>(ws + w.v16);
  const uint16_t* src[1] = {v};
  uint16_t* dst[1] = {v16};
  const size_t n[1] = {(size_t)B * Hkv * Lk * D};
  int* work = reinterpret_cast<int*>(ws + w.work);
  if (launch("convert_f16", s, [&] { return swa::launch_convert_f16(src, dst, n, 1, status, s, work); }) !=
      cudaSuccess)
    return SWA_ERR_CUDA;
  if (launch("fwd_tc", s, [&] { return swa::launch_fwd_tc(g, q, k, v16, o, lse, work, status, s); }) != cudaSuccess)
    return SWA_ERR_CUDA;
  return SWA_OK;
}


// The backward on a shape-checked geometry (the tail of swa_attn_bwd_ex and
// swa_attn_bwd_prefix).
static int bwd_run(const swa::Geom& g, const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, const float* o,
                   const float* lse, const swa_bf16* dO, float* dq, float* dk, float* dv, void* workspace,
                   size_t workspace_bytes, void* stream, float* dsinks = nullptr) {
  const int B = g.B, Hq = g.Hq, Hkv = g.Hkv, Lq = g.Lq, Lk = g.L, D = g.D;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 16) ||
      !aligned(dO, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(workspace, 256))
    return SWA_ERR_MISALIGNED;
  const size_t need = bwd_tc_ws_layout(B, Hq, Hkv, Lq, Lk, D).total;
  if (!workspace || workspace_bytes < need) return SWA_ERR_WORKSPACE;
  int rc = check_device();
  if (rc) return rc;
  if (D == 512 && (rc = check_scratch_layout(kScratchBwd512)) != SWA_OK) return rc;
  if (D == 256 && (rc = check_scratch_layout(kScratchBwd256)) != SWA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = status_ptr_for_current_device(&rc);
  if (!status) return rc;
  const BwdTcWs w = bwd_tc_ws_layout(B, Hq, Hkv, Lq, Lk, D);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  float* stats = reinterpret_cast<float*>(ws + w.stats);
  uint16_t* q16 = reinterpret_cast<uint16_t*>(ws + w.q16);
  uint16_t* k16 = reinterpret_cast<uint16_t*>(ws + w.k16);
  uint16_t* v16 = reinterpret_cast<uint16_t*>(ws + w.v16);
  uint16_t* g16 = reinterpret_cast<uint16_t*>(ws + w.g16);
  // max |dO| first: the prep scales dO's fp16 copy by a power of two from it
  if (launch("bwd_dscale", s, [&] { return swa::launch_bwd_dscale(g, w.Lpad, dO, stats, s); }) != cudaSuccess)
    return SWA_ERR_CUDA;
  if (launch("bwd_prep", s, [&] {
        return swa::launch_bwd_prep(g, w.Lpad, q, k, v, dO, o, lse, q16, k16, v16, g16, stats, status, s);
      }) != cudaSuccess)
    return SWA_ERR_CUDA;
  // attention sinks: their gradient needs only the row statistics
  if (g.sinks &&
      launch("bwd_sink_grad", s, [&] { return swa::launch_sink_grad(g, w.Lpad, stats, dsinks, s); }) != cudaSuccess)
    return SWA_ERR_CUDA;
  // The dK/dV and dQ passes read the same inputs, write disjoint outputs
  // and run side by side.
  if (D == 512) {
    // Both passes are persistent (as many clusters as fit, looping over work
    // items).  dK/dV goes first and takes the SMs its clusters can use; dQ,
    // launched after it on the same stream as a programmatic dependent,
    // starts on the SMs it leaves and takes over those its clusters free as
    // its work runs out.
    const cudaError_t e = launch_overlapped(
        "bwd_dkdv_tc", "bwd_dq_tc", s,
        [&] { return swa::launch_bwd_dkdv_tc(g, q16, k16, v16, g16, stats, w.Lpad, dk, dv, status, s); },
        [&] { return swa::launch_bwd_dq_tc(g, q16, k16, v16, g16, stats, w.Lpad, dq, status, s); });
    return e == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
  }
  // Up to head dim 256: dK/dV on the side stream (forked after the prep),
  // whose higher priority gives its waiting CTAs the SMs that free up first,
  // dQ on the caller's stream, which then waits for the side stream.
  SideStream* side = side_stream_for_current_device();
  if (!side) return SWA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(side->mu);
  cudaStream_t t = side->stream;
  if (cudaEventRecord(side->fork, s) != cudaSuccess || cudaStreamWaitEvent(t, side->fork, 0) != cudaSuccess)
    return SWA_ERR_CUDA;
  const cudaError_t e_dkdv = launch("bwd_dkdv_tc", t, [&] {
    return swa::launch_bwd_dkdv_tc(g, q16, k16, v16, g16, stats, w.Lpad, dk, dv, status, t);
  });
  const cudaError_t e_dq = launch("bwd_dq_tc", s, [&] {
    return swa::launch_bwd_dq_tc(g, q16, k16, v16, g16, stats, w.Lpad, dq, status, s);
  });
  // the join is recorded even after a failed launch, so that the caller's
  // stream never runs ahead of work already queued on the side stream
  if (cudaEventRecord(side->join, t) != cudaSuccess || cudaStreamWaitEvent(s, side->join, 0) != cudaSuccess)
    return SWA_ERR_CUDA;
  if (e_dkdv != cudaSuccess || e_dq != cudaSuccess) return SWA_ERR_CUDA;
  return SWA_OK;
}


extern "C" {

int swa_attn_version(void) { return 100; }

const char* swa_attn_strerror(int code) {
  switch (code) {
    case SWA_OK: return "success";
    case SWA_ERR_NULL_POINTER: return "a required pointer is NULL";
    case SWA_ERR_BAD_SHAPE: return "B, Hq, Hkv and Lq must be >= 1, and Lk >= Lq";
    case SWA_ERR_BAD_GROUPS: return "Hq must be a multiple of Hkv";
    case SWA_ERR_BAD_HEAD_DIM: return "head dim D must be 64, 128, 256 or 512";
    case SWA_ERR_BAD_WINDOW: return "window must be >= 0 (0 = no window)";
    case SWA_ERR_BAD_SCALE: return "scale must be finite";
    case SWA_ERR_MISALIGNED: return "tensors must be 16-byte aligned and the workspace 256-byte aligned";
    case SWA_ERR_WORKSPACE: return "workspace smaller than the size query returned";
    case SWA_ERR_CUDA: return "CUDA runtime or launch error";
    case SWA_ERR_TOO_LARGE: return "sizes exceed the supported range";
    case SWA_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait expired";
    case SWA_ERR_UNSUPPORTED_DEVICE: return "current device is not an sm_103 GPU";
    case SWA_ERR_FP16_RANGE: return "an input magnitude overflowed the fp16 operand copy (|x| > 65504)";
    case SWA_ERR_BAD_PLAN:
      return "shared-prefix plan needs prompt_len >= 0, chosen_len >= 0 and prompt_len + chosen_len <= L";
    case SWA_ERR_SCRATCH_LAYOUT:
      return "head dim 512 needs at most one CTA per SM and SM ids below 192 for its per-SM tile scratch";
    case SWA_ERR_NOALLOC_LIMIT:
      return "B*Hq*L exceeds the fixed scratch of swa_attn_bwd_noalloc (2,097,152 rows); use swa_attn_bwd";
    default: return "unknown error code";
  }
}

size_t swa_attn_fwd_workspace_bytes_ex(int B, int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Lq < 1 || Lk < Lq || Hq % Hkv != 0 || window < 0 || !swa::fwd_tc_supported(D))
    return 0;
  return fwd_need(make_geom(B, Hq, Hkv, Lq, Lk, D, window, causal, 1.f));
}

size_t swa_attn_bwd_workspace_bytes_ex(int B, int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal) {
  (void)window;
  (void)causal;
  if (B < 1 || Hq < 1 || Hkv < 1 || Lq < 1 || Lk < Lq) return 0;
  if (swa::bwd_tc_supported(D)) return bwd_tc_ws_layout(B, Hq, Hkv, Lq, Lk, D).total;
  return bwd_delta_bytes(B, Hq, Lq);
}

size_t swa_attn_fwd_workspace_bytes(int B, int Hq, int Hkv, int L, int D, int window) {
  return swa_attn_fwd_workspace_bytes_ex(B, Hq, Hkv, L, L, D, window, 1);
}

size_t swa_attn_bwd_workspace_bytes(int B, int Hq, int Hkv, int L, int D, int window) {
  return swa_attn_bwd_workspace_bytes_ex(B, Hq, Hkv, L, L, D, window, 1);
}

int swa_attn_fwd_ex(const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, float* o, float* lse, int B, int Hq,
                    int Hkv, int Lq, int Lk, int D, int window, int causal, float scale, void* workspace,
                    size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !lse) return SWA_ERR_NULL_POINTER;
  const int rc = check_shape(B, Hq, Hkv, Lq, Lk, D, window, scale);
  if (rc) return rc;
  return fwd_run(make_geom(B, Hq, Hkv, Lq, Lk, D, window, causal, scale), q, k, v, o, lse, workspace,
                 workspace_bytes, stream);
}

int swa_attn_fwd(const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, float* o, float* lse, int B, int Hq,
                 int Hkv, int L, int D, int window, float scale, void* workspace, size_t workspace_bytes,
                 void* stream) {
  return swa_attn_fwd_ex(q, k, v, o, lse, B, Hq, Hkv, L, L, D, window, 1, scale, workspace, workspace_bytes,
                         stream);
}

int swa_attn_bwd_ex(const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, const float* o, const float* lse,
                    const swa_bf16* dO, float* dq, float* dk, float* dv, int B, int Hq, int Hkv, int Lq, int Lk,
                    int D, int window, int causal, float scale, void* workspace, size_t workspace_bytes,
                    void* stream) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return SWA_ERR_NULL_POINTER;
  const int rc = check_shape(B, Hq, Hkv, Lq, Lk, D, window, scale);
  if (rc) return rc;
  return bwd_run(make_geom(B, Hq, Hkv, Lq, Lk, D, window, causal, scale), q, k, v, o, lse, dO, dq, dk, dv,
                 workspace, workspace_bytes, stream);
}

int swa_attn_bwd(const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, const float* o, const float* lse,
                 const swa_bf16* dO, float* dq, float* dk, float* dv, int B, int Hq, int Hkv, int L, int D,
                 int window, float scale, void* workspace, size_t workspace_bytes, void* stream) {
  return swa_attn_bwd_ex(q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, L, L, D, window, 1, scale, workspace,
                         workspace_bytes, stream);
}

size_t swa_attn_fwd_workspace_bytes_prefix(int B, int Hq, int Hkv, int L, int D, int window, int prompt_len,
                                            int chosen_len) {
  if (B < 1 || Hq < 1 || Hkv < 1 || L < 1 || Hq % Hkv != 0 || window < 0 || !swa::fwd_tc_supported(D) ||
      check_plan(L, prompt_len, chosen_len))
    return 0;
  return fwd_need(make_plan_geom(B, Hq, Hkv, L, D, window, prompt_len, chosen_len, 1.f));
}

size_t swa_attn_bwd_workspace_bytes_prefix(int B, int Hq, int Hkv, int L, int D, int window, int prompt_len,
                                            int chosen_len) {
  if (check_plan(L, prompt_len, chosen_len)) return 0;
  return swa_attn_bwd_workspace_bytes(B, Hq, Hkv, L, D, window);
}

int swa_attn_fwd_prefix(const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, float* o, float* lse, int B,
                        int Hq, int Hkv, int L, int D, int window, int prompt_len, int chosen_len, float scale,
                        void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !lse) return SWA_ERR_NULL_POINTER;
  int rc = check_shape(B, Hq, Hkv, L, L, D, window, scale);
  if (rc) return rc;
  if ((rc = check_plan(L, prompt_len, chosen_len))) return rc;
  return fwd_run(make_plan_geom(B, Hq, Hkv, L, D, window, prompt_len, chosen_len, scale), q, k, v, o, lse,
                 workspace, workspace_bytes, stream);
}

int swa_attn_bwd_prefix(const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, const float* o, const float* lse,
                        const swa_bf16* dO, float* dq, float* dk, float* dv, int B, int Hq, int Hkv, int L, int D,
                        int window, int prompt_len, int chosen_len, float scale, void* workspace,
                        size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return SWA_ERR_NULL_POINTER;
  int rc = check_shape(B, Hq, Hkv, L, L, D, window, scale);
  if (rc) return rc;
  if ((rc = check_plan(L, prompt_len, chosen_len))) return rc;
  return bwd_run(make_plan_geom(B, Hq, Hkv, L, D, window, prompt_len, chosen_len, scale), q, k, v, o, lse, dO, dq,
                 dk, dv, workspace, workspace_bytes, stream);
}

int swa_attn_fwd_sinks(const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, const float* sinks, float* o,
                       float* lse, int B, int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal, float scale,
                       void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !sinks || !o || !lse) return SWA_ERR_NULL_POINTER;
  const int rc = check_shape(B, Hq, Hkv, Lq, Lk, D, window, scale);
  if (rc) return rc;
  if (!aligned(sinks, 4)) return SWA_ERR_MISALIGNED;
  swa::Geom g = make_geom(B, Hq, Hkv, Lq, Lk, D, window, causal, scale);
  g.sinks = sinks;
  return fwd_run(g, q, k, v, o, lse, workspace, workspace_bytes, stream);
}

int swa_attn_bwd_sinks(const swa_bf16* q, const swa_bf16* k, const swa_bf16* v, const float* sinks, const float* o,
                       const float* lse, const swa_bf16* dO, float* dq, float* dk, float* dv, float* dsinks, int B,
                       int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal, float scale, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !sinks || !o || !lse || !dO || !dq || !dk || !dv || !dsinks) return SWA_ERR_NULL_POINTER;
  const int rc = check_shape(B, Hq, Hkv, Lq, Lk, D, window, scale);
  if (rc) return rc;
  if (!aligned(sinks, 4) || !aligned(dsinks, 4)) return SWA_ERR_MISALIGNED;
  swa::Geom g = make_geom(B, Hq, Hkv, Lq, Lk, D, window, causal, scale);
  g.sinks = sinks;
  return bwd_run(g, q, k, v, o, lse, dO, dq, dk, dv, workspace, workspace_bytes, stream, dsinks);
}

int swa_attn_selftest_timeout(void* stream) {
  int rc = check_device();
  if (rc != SWA_OK) return rc;
  int err = SWA_OK;
  int* p = status_ptr_for_current_device(&err);
  if (!p) return err;
  // about 1 ms at the maximum SM clock
  if (swa::launch_selftest_timeout(p, 2000000LL, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SWA_ERR_CUDA;
  return SWA_OK;
}

int swa_attn_get_status(void* stream) {
  int err = SWA_OK;
  int* p = status_ptr_for_current_device(&err);
  if (!p) return err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int host = 0;
  if (cudaMemcpyAsync(&host, p, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return SWA_ERR_CUDA;
  if (cudaMemsetAsync(p, 0, sizeof(int), s) != cudaSuccess) return SWA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SWA_ERR_CUDA;
  return host;
}

int swa_attn_profile_begin(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (auto& r : g_prof_recs) {
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  g_prof_recs.clear();
  g_prof_on = true;
  return SWA_OK;
}

int swa_attn_profile_end(swa_attn_kernel_time* out, int max_entries, int* n_out) {
  std::vector<ProfRec> recs;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_on = false;
    recs.swap(g_prof_recs);
  }
  int rc = SWA_OK;
  std::vector<swa_attn_kernel_time> agg;
  for (auto& r : recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
      rc = SWA_ERR_CUDA;
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
    size_t idx = 0;
    while (idx < agg.size() && strncmp(agg[idx].name, r.name.c_str(), sizeof(agg[idx].name)) != 0) ++idx;
    if (idx == agg.size()) {
      swa_attn_kernel_time t;
      memset(&t, 0, sizeof t);
      strncpy(t.name, r.name.c_str(), sizeof(t.name) - 1);
      agg.push_back(t);
    }
    agg[idx].launches += 1;
    agg[idx].total_ms += ms;
  }
  int n = 0;
  for (size_t i = 0; i < agg.size() && n < max_entries; ++i) {
    if (out) out[n] = agg[i];
    ++n;
  }
  if (n_out) *n_out = n;
  return rc;
}

}  // extern "C"
