// Internal interface between the C-ABI translation unit and the kernel
// translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>

namespace swa {

// Problem geometry shared by every kernel.
struct Geom {
  int B, Hq, Hkv, L, D, W, G;  // G = Hq / Hkv; W = 0 means plain causal
  float scale;                 // softmax scale applied to q . k
};

// Device-side status codes latched into the per-device status word.
enum : int { kStatusOk = 0, kStatusTimeout = -11, kStatusFp16Range = -14 };

// ---- SIMT kernels (fp32 arithmetic on bf16 inputs; any D in {64..512}) ----
cudaError_t launch_fwd_simt(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                            float* o, float* lse, cudaStream_t s);
cudaError_t launch_delta(const Geom& g, const float* o, const uint16_t* dO, float* delta, cudaStream_t s);
cudaError_t launch_bwd_dkdv_simt(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                 const uint16_t* dO, const float* lse, const float* delta, float* dk,
                                 float* dv, cudaStream_t s);
cudaError_t launch_bwd_dq_simt(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               const uint16_t* dO, const float* lse, const float* delta, float* dq,
                               cudaStream_t s);

// ---- tensor-core path (tcgen05 + TMA + TMEM), fp16 operand copies ----
// bf16 -> fp16 copies of up to four tensors (n[i] elements, multiples of 8);
// latches kStatusFp16Range in *status if a finite input overflows fp16.
cudaError_t launch_convert_f16(const uint16_t* const* src, uint16_t* const* dst, const size_t* n, int count,
                               int* status, cudaStream_t s);
// One CTA whose bounded wait on a barrier nothing completes runs out after
// limit_cycles and latches kStatusTimeout in *status.
cudaError_t launch_selftest_timeout(int* status, long long limit_cycles, cudaStream_t s);
bool fwd_tc_supported(int D);
// Head dim 512: 2-CTA cluster forward (tc_fwd512.cu).
cudaError_t launch_fwd_tc512(const Geom& g, const uint16_t* q16, const uint16_t* k16, const uint16_t* v16, float* o,
                             float* lse, int* status, cudaStream_t s);
cudaError_t launch_fwd_tc(const Geom& g, const uint16_t* q16, const uint16_t* k16, const uint16_t* v16, float* o,
                          float* lse, int* status, cudaStream_t s);

// 3-D fp16 tensor map over [heads, L, D] with a 64 x box_rows box and
// 128-byte swizzle (rows at or beyond L read as zero).
cudaError_t make_tmap_f16(CUtensorMap* m, const void* ptr, int D, int L, int heads, int box_rows);
// The same tensor as a 4-D map whose box (64, box_rows, nchunk, 1) loads
// nchunk 64-column chunks (consecutive [box_rows x 128 B] swizzled blocks)
// with one TMA instruction; coordinates (0, row, first chunk, head).
cudaError_t make_tmap_f16_chunks(CUtensorMap* m, const void* ptr, int D, int L, int heads, int box_rows,
                                 int nchunk);

bool bwd_tc_supported(int D);
// Padded row count of the backward's row-statistics array.
int bwd_stats_lpad(int L);
// Two planes of B * Hq * Lpad floats: stats[bh * Lpad + i] = lse_i * log2(e),
// stats[(B * Hq + bh) * Lpad + i] = dO_i . o_i; zero for i >= L.
cudaError_t launch_rowstats(const Geom& g, int Lpad, const float* o, const uint16_t* dO, const float* lse,
                            float* stats, cudaStream_t s);
cudaError_t launch_bwd_dkdv_tc(const Geom& g, const uint16_t* q16, const uint16_t* k16, const uint16_t* v16,
                               const uint16_t* g16, const float* stats, int Lpad, float* dk, float* dv,
                               int* status, cudaStream_t s);
// Head dim 512: thread-block-cluster kernels (tc_bwd512.cu).
cudaError_t launch_bwd_dkdv_tc512(const Geom& g, const uint16_t* q16, const uint16_t* k16, const uint16_t* v16,
                                  const uint16_t* g16, const float* stats, int Lpad, float* dk, float* dv,
                                  int* status, cudaStream_t s);
cudaError_t launch_bwd_dq_tc512(const Geom& g, const uint16_t* q16, const uint16_t* k16, const uint16_t* v16,
                                const uint16_t* g16, const float* stats, int Lpad, float* dq, int* status,
                                cudaStream_t s);
cudaError_t launch_bwd_dq_tc(const Geom& g, const uint16_t* q16, const uint16_t* k16, const uint16_t* v16,
                             const uint16_t* g16, const float* stats, int Lpad, float* dq, int* status,
                             cudaStream_t s);

}  // namespace swa
