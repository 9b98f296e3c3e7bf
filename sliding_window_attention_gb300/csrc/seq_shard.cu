// Sequence sharding: the reduction that returns halo key gradients to the
// rank that owns those keys.
//
// When a sequence is split into contiguous chunks, one per rank, the queries
// of a chunk see keys of earlier chunks (the W - 1 keys behind the chunk for
// a causal window of W, every earlier key without a window).  Each rank runs
// the attention of its queries over [halo; own keys] (queries a suffix of the
// keys), so its backward produces dK and dV rows for the halo keys too.
// Those rows are partial sums of the owner's gradients: the owner adds them
// into its own dK and dV.  This file holds that add.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/swa_attn.h"

namespace {

// dst[bh, row0 + r, :] += src[bh, r, :] for r < nrows; D is a multiple of 4,
// so each thread adds one 16-byte vector, grid-stride.
__global__ void __launch_bounds__(256) add_rows_kernel(float* __restrict__ dst, const float* __restrict__ src,
                                                        long long n4, int nrows, int dst_rows, int row0, int d4) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < n4; idx += stride) {
    const long long row = idx / d4;  // bh * nrows + r
    const int c = (int)(idx - row * d4);
    const long long bh = row / nrows;
    const int r = (int)(row - bh * nrows);
    float4* d = reinterpret_cast<float4*>(dst) + ((bh * dst_rows + row0 + r) * d4 + c);
    const float4 s = __ldg(reinterpret_cast<const float4*>(src) + idx);
    float4 v = *d;
    v.x += s.x;
    v.y += s.y;
    v.z += s.z;
    v.w += s.w;
    *d = v;
  }
}

}  // namespace

extern "C" int swa_attn_add_rows_f32(float* dst, const float* src, int BH, int dst_rows, int row0, int nrows, int D,
                                     void* stream) {
  if (!dst || !src) return SWA_ERR_NULL_POINTER;
  if (BH < 1 || dst_rows < 1 || nrows < 0 || row0 < 0 || (long long)row0 + nrows > dst_rows || D < 4 || D % 4)
    return SWA_ERR_BAD_SHAPE;
  if ((reinterpret_cast<uintptr_t>(dst) & 15u) || (reinterpret_cast<uintptr_t>(src) & 15u)) return SWA_ERR_MISALIGNED;
  if (nrows == 0) return SWA_OK;
  const long long n4 = (long long)BH * nrows * (D / 4);
  long long blocks = (n4 + 255) / 256;
  if (blocks > 152LL * 8) blocks = 152LL * 8;
  add_rows_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(dst, src, n4, nrows, dst_rows,
                                                                                   row0, D / 4);
  return cudaGetLastError() == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}
