// SIMT kernels: forward (o, lse), the Delta row term, the key-outer dK/dV
// pass and the query-outer dQ pass, in plain fp32 CUDA-core arithmetic on
// bf16 inputs.  They follow the same band / tile rules as the tensor-core
// kernels and serve head dims that those do not cover.
//
// Tile rules ("Lab 028 lab detail: Off NVIDIA, you fix the platform
// yourself", "What I changed, in plain terms" items 3-5): a query tile
// visits only key tiles that intersect its band, a key tile only query tiles
// whose band reaches it; inside an edge tile P is zeroed where j > i or
// i - j >= window.  dQ is produced by its own pass (no read-modify-write of a
// partially initialised buffer, item 5a) and dK/dV are written for every key
// row, visited or not.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "swa_internal.h"

namespace swa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kThreads = 256;
constexpr int kPad = 8;  // bf16 elements of padding per shared-memory row (16 bytes)

__device__ __forceinline__ bool in_band(int i, int j, int W) { return j <= i && (W == 0 || i - j < W); }

// Two packed bf16 (low half first) -> two floats.  bf16 -> fp32 is exact.
__device__ __forceinline__ float2 bf2f(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// rows x D bf16 from global (stride D) into shared memory (stride D + kPad);
// rows at or beyond `valid` are zero-filled.
template <int D>
__device__ __forceinline__ void load_rows(uint16_t* __restrict__ sm, const uint16_t* __restrict__ gm, int rows,
                                          int valid) {
  constexpr int kChunks = D / 8;
  for (int idx = threadIdx.x; idx < rows * kChunks; idx += kThreads) {
    const int r = idx / kChunks, c = idx - r * kChunks;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (r < valid) val = __ldg(reinterpret_cast<const uint4*>(gm + (size_t)r * D) + c);
    *reinterpret_cast<uint4*>(sm + r * (D + kPad) + c * 8) = val;
  }
}

// ---------------------------------------------------------------------------
// Forward: one CTA per (query tile of BM rows, query head, batch).
template <int D, int BM, int BN>
__global__ void __launch_bounds__(kThreads) fwd_simt_kernel(Geom g, const uint16_t* __restrict__ q,
                                                            const uint16_t* __restrict__ k,
                                                            const uint16_t* __restrict__ v, float* __restrict__ o,
                                                            float* __restrict__ lse) {
  constexpr int TPR = kThreads / BM;  // threads per query row
  constexpr int CPT = BN / TPR;       // score columns per thread
  constexpr int DP = D / 2 / TPR;     // output column pairs per thread
  constexpr int LDS = D + kPad;
  extern __shared__ __align__(16) unsigned char smem[];
  uint16_t* Qs = reinterpret_cast<uint16_t*>(smem);
  uint16_t* Ks = Qs + BM * LDS;
  uint16_t* Vs = Ks + BN * LDS;
  float* Ps = reinterpret_cast<float*>(Vs + BN * LDS);  // [BM][BN + 1]

  const int i0 = blockIdx.x * BM, h = blockIdx.y, b = blockIdx.z;
  const int kvh = h / g.G;
  const int r = threadIdx.x / TPR, c = threadIdx.x % TPR;
  const int i = i0 + r;
  const size_t qbase = (size_t)(b * g.Hq + h) * g.L * D;
  const size_t kbase = (size_t)(b * g.Hkv + kvh) * g.L * D;
  load_rows<D>(Qs, q + qbase + (size_t)i0 * D, BM, min(BM, g.L - i0));

  const float sl2 = g.scale * kLog2e;
  float m = -INFINITY, l = 0.f;
  float acc[2 * DP];
#pragma unroll
  for (int u = 0; u < 2 * DP; ++u) acc[u] = 0.f;

  const int ihi = min(i0 + BM, g.L) - 1;
  const int jlo = g.W > 0 ? max(0, i0 - g.W + 1) : 0;
  for (int t = jlo / BN; t <= ihi / BN; ++t) {
    const int j0 = t * BN;
    __syncthreads();
    load_rows<D>(Ks, k + kbase + (size_t)j0 * D, BN, min(BN, g.L - j0));
    load_rows<D>(Vs, v + kbase + (size_t)j0 * D, BN, min(BN, g.L - j0));
    __syncthreads();

    float s[CPT];
#pragma unroll
    for (int mm = 0; mm < CPT; ++mm) s[mm] = 0.f;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(Qs + r * LDS);
#pragma unroll 4
    for (int d2 = 0; d2 < D / 2; ++d2) {
      const float2 qa = bf2f(qrow[d2]);
#pragma unroll
      for (int mm = 0; mm < CPT; ++mm) {
        const float2 kb = bf2f(reinterpret_cast<const uint32_t*>(Ks + (c + TPR * mm) * LDS)[d2]);
        s[mm] = fmaf(qa.x, kb.x, s[mm]);
        s[mm] = fmaf(qa.y, kb.y, s[mm]);
      }
    }
    float tmax = -INFINITY;
#pragma unroll
    for (int mm = 0; mm < CPT; ++mm) {
      const int j = j0 + c + TPR * mm;
      const bool ok = i < g.L && j < g.L && in_band(i, j, g.W);
      s[mm] = ok ? s[mm] * sl2 : -INFINITY;
      tmax = fmaxf(tmax, s[mm]);
    }
#pragma unroll
    for (int off = 1; off < TPR; off <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
    const float m_new = fmaxf(m, tmax);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = exp2f(m - m_use);
    float psum = 0.f;
#pragma unroll
    for (int mm = 0; mm < CPT; ++mm) {
      const float p = exp2f(s[mm] - m_use);
      Ps[r * (BN + 1) + c + TPR * mm] = p;
      psum += p;
    }
#pragma unroll
    for (int off = 1; off < TPR; off <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
    l = l * alpha + psum;
    m = m_new;
#pragma unroll
    for (int u = 0; u < 2 * DP; ++u) acc[u] *= alpha;
    __syncwarp();
    const float* prow = Ps + r * (BN + 1);
#pragma unroll 2
    for (int jj = 0; jj < BN; ++jj) {
      const float p = prow[jj];
      const uint32_t* vrow = reinterpret_cast<const uint32_t*>(Vs + jj * LDS);
#pragma unroll
      for (int u = 0; u < DP; ++u) {
        const float2 vv = bf2f(vrow[c + TPR * u]);
        acc[2 * u] = fmaf(p, vv.x, acc[2 * u]);
        acc[2 * u + 1] = fmaf(p, vv.y, acc[2 * u + 1]);
      }
    }
    __syncwarp();
  }
  if (i < g.L) {
    const float inv = 1.f / l;
    float2* orow = reinterpret_cast<float2*>(o + qbase + (size_t)i * D);
#pragma unroll
    for (int u = 0; u < DP; ++u) orow[c + TPR * u] = make_float2(acc[2 * u] * inv, acc[2 * u + 1] * inv);
    if (c == 0) lse[(size_t)(b * g.Hq + h) * g.L + i] = (m + log2f(l)) / kLog2e;
  }
}

// ---------------------------------------------------------------------------
// Delta_i = dO_i . o_i: one warp per row.
__global__ void __launch_bounds__(kThreads) delta_kernel(long rows, int D, const float* __restrict__ o,
                                                         const uint16_t* __restrict__ dO,
                                                         float* __restrict__ delta) {
  const long row = ((long)blockIdx.x * kThreads + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (row >= rows) return;
  const float* orow = o + row * D;
  const uint16_t* grow = dO + row * D;
  float acc = 0.f;
  for (int d = lane * 4; d < D; d += 128) {
    const float4 ov = *reinterpret_cast<const float4*>(orow + d);
    const uint2 gv = *reinterpret_cast<const uint2*>(grow + d);
    const float2 g01 = bf2f(gv.x), g23 = bf2f(gv.y);
    acc = fmaf(ov.x, g01.x, acc);
    acc = fmaf(ov.y, g01.y, acc);
    acc = fmaf(ov.z, g23.x, acc);
    acc = fmaf(ov.w, g23.y, acc);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) delta[row] = acc;
}

// ---------------------------------------------------------------------------
// dK / dV: one CTA per (key tile of BN rows, kv head, batch); loops over the
// group's query heads and the query tiles of BM rows whose band reaches it.
template <int D, int BN, int BM>
__global__ void __launch_bounds__(kThreads) dkdv_simt_kernel(Geom g, const uint16_t* __restrict__ q,
                                                             const uint16_t* __restrict__ k,
                                                             const uint16_t* __restrict__ v,
                                                             const uint16_t* __restrict__ dO,
                                                             const float* __restrict__ lse,
                                                             const float* __restrict__ delta, float* __restrict__ dk,
                                                             float* __restrict__ dv) {
  constexpr int TPR = kThreads / BN;  // threads per key row
  constexpr int CPT = BM / TPR;       // query columns per thread
  constexpr int DP = D / 2 / TPR;     // output column pairs per thread
  constexpr int LDS = D + kPad;
  extern __shared__ __align__(16) unsigned char smem[];
  uint16_t* Ks = reinterpret_cast<uint16_t*>(smem);
  uint16_t* Vs = Ks + BN * LDS;
  uint16_t* Qs = Vs + BN * LDS;
  uint16_t* Gs = Qs + BM * LDS;
  float* Ps = reinterpret_cast<float*>(Gs + BM * LDS);  // [BN][BM + 1]
  float* Ss = Ps + BN * (BM + 1);                        // [BN][BM + 1]
  float* lse_s = Ss + BN * (BM + 1);                     // [BM], pre-multiplied by log2(e)
  float* dl_s = lse_s + BM;                              // [BM]

  const int j0 = blockIdx.x * BN, kvh = blockIdx.y, b = blockIdx.z;
  const int r = threadIdx.x / TPR, c = threadIdx.x % TPR;
  const int j = j0 + r;
  const size_t kbase = (size_t)(b * g.Hkv + kvh) * g.L * D;
  load_rows<D>(Ks, k + kbase + (size_t)j0 * D, BN, min(BN, g.L - j0));
  load_rows<D>(Vs, v + kbase + (size_t)j0 * D, BN, min(BN, g.L - j0));

  const float sl2 = g.scale * kLog2e;
  float adk[2 * DP], adv[2 * DP];
#pragma unroll
  for (int u = 0; u < 2 * DP; ++u) adk[u] = adv[u] = 0.f;

  const int jhi = min(j0 + BN, g.L) - 1;
  const int ihi = g.W > 0 ? min(g.L - 1, jhi + g.W - 1) : g.L - 1;
  for (int gi = 0; gi < g.G; ++gi) {
    const int h = kvh * g.G + gi;
    const size_t qbase = (size_t)(b * g.Hq + h) * g.L * D;
    const size_t rbase = (size_t)(b * g.Hq + h) * g.L;
    for (int t = j0 / BM; t <= ihi / BM; ++t) {
      const int i0 = t * BM;
      __syncthreads();
      load_rows<D>(Qs, q + qbase + (size_t)i0 * D, BM, min(BM, g.L - i0));
      load_rows<D>(Gs, dO + qbase + (size_t)i0 * D, BM, min(BM, g.L - i0));
      for (int x = threadIdx.x; x < BM; x += kThreads) {
        const bool ok = i0 + x < g.L;
        lse_s[x] = ok ? lse[rbase + i0 + x] * kLog2e : 0.f;
        dl_s[x] = ok ? delta[rbase + i0 + x] : 0.f;
      }
      __syncthreads();

      float s[CPT], dp[CPT];
#pragma unroll
      for (int mm = 0; mm < CPT; ++mm) s[mm] = dp[mm] = 0.f;
      const uint32_t* krow = reinterpret_cast<const uint32_t*>(Ks + r * LDS);
      const uint32_t* vrow = reinterpret_cast<const uint32_t*>(Vs + r * LDS);
#pragma unroll 2
      for (int d2 = 0; d2 < D / 2; ++d2) {
        const float2 kk = bf2f(krow[d2]);
        const float2 vv = bf2f(vrow[d2]);
#pragma unroll
        for (int mm = 0; mm < CPT; ++mm) {
          const int ci = c + TPR * mm;
          const float2 qa = bf2f(reinterpret_cast<const uint32_t*>(Qs + ci * LDS)[d2]);
          const float2 ga = bf2f(reinterpret_cast<const uint32_t*>(Gs + ci * LDS)[d2]);
          s[mm] = fmaf(kk.x, qa.x, fmaf(kk.y, qa.y, s[mm]));
          dp[mm] = fmaf(vv.x, ga.x, fmaf(vv.y, ga.y, dp[mm]));
        }
      }
#pragma unroll
      for (int mm = 0; mm < CPT; ++mm) {
        const int ci = c + TPR * mm, i = i0 + ci;
        const bool ok = i < g.L && j < g.L && in_band(i, j, g.W);
        const float p = ok ? exp2f(fmaf(s[mm], sl2, -lse_s[ci])) : 0.f;
        Ps[r * (BM + 1) + ci] = p;
        Ss[r * (BM + 1) + ci] = p * (dp[mm] - dl_s[ci]);
      }
      __syncwarp();
      const float* prow = Ps + r * (BM + 1);
      const float* srow = Ss + r * (BM + 1);
#pragma unroll 2
      for (int ci = 0; ci < BM; ++ci) {
        const float p = prow[ci], ds = srow[ci];
        const uint32_t* qr = reinterpret_cast<const uint32_t*>(Qs + ci * LDS);
        const uint32_t* gr = reinterpret_cast<const uint32_t*>(Gs + ci * LDS);
#pragma unroll
        for (int u = 0; u < DP; ++u) {
          const float2 qa = bf2f(qr[c + TPR * u]);
          const float2 ga = bf2f(gr[c + TPR * u]);
          adv[2 * u] = fmaf(p, ga.x, adv[2 * u]);
          adv[2 * u + 1] = fmaf(p, ga.y, adv[2 * u + 1]);
          adk[2 * u] = fmaf(ds, qa.x, adk[2 * u]);
          adk[2 * u + 1] = fmaf(ds, qa.y, adk[2 * u + 1]);
        }
      }
      __syncwarp();
    }
  }
  if (j < g.L) {
    float2* dkrow = reinterpret_cast<float2*>(dk + kbase + (size_t)j * D);
    float2* dvrow = reinterpret_cast<float2*>(dv + kbase + (size_t)j * D);
#pragma unroll
    for (int u = 0; u < DP; ++u) {
      dkrow[c + TPR * u] = make_float2(adk[2 * u] * g.scale, adk[2 * u + 1] * g.scale);
      dvrow[c + TPR * u] = make_float2(adv[2 * u], adv[2 * u + 1]);
    }
  }
}

// ---------------------------------------------------------------------------
// dQ: one CTA per (query tile of BM rows, query head, batch); recomputes S,
// P, dP and dS over the key tiles of its band.
template <int D, int BM, int BN>
__global__ void __launch_bounds__(kThreads) dq_simt_kernel(Geom g, const uint16_t* __restrict__ q,
                                                           const uint16_t* __restrict__ k,
                                                           const uint16_t* __restrict__ v,
                                                           const uint16_t* __restrict__ dO,
                                                           const float* __restrict__ lse,
                                                           const float* __restrict__ delta, float* __restrict__ dq) {
  constexpr int TPR = kThreads / BM;
  constexpr int CPT = BN / TPR;
  constexpr int DP = D / 2 / TPR;
  constexpr int LDS = D + kPad;
  extern __shared__ __align__(16) unsigned char smem[];
  uint16_t* Qs = reinterpret_cast<uint16_t*>(smem);
  uint16_t* Gs = Qs + BM * LDS;
  uint16_t* Ks = Gs + BM * LDS;
  uint16_t* Vs = Ks + BN * LDS;
  float* Ss = reinterpret_cast<float*>(Vs + BN * LDS);  // [BM][BN + 1]

  const int i0 = blockIdx.x * BM, h = blockIdx.y, b = blockIdx.z;
  const int kvh = h / g.G;
  const int r = threadIdx.x / TPR, c = threadIdx.x % TPR;
  const int i = i0 + r;
  const size_t qbase = (size_t)(b * g.Hq + h) * g.L * D;
  const size_t kbase = (size_t)(b * g.Hkv + kvh) * g.L * D;
  const size_t rbase = (size_t)(b * g.Hq + h) * g.L;
  load_rows<D>(Qs, q + qbase + (size_t)i0 * D, BM, min(BM, g.L - i0));
  load_rows<D>(Gs, dO + qbase + (size_t)i0 * D, BM, min(BM, g.L - i0));
  const float lse_l2 = i < g.L ? lse[rbase + i] * kLog2e : 0.f;
  const float dl = i < g.L ? delta[rbase + i] : 0.f;

  const float sl2 = g.scale * kLog2e;
  float acc[2 * DP];
#pragma unroll
  for (int u = 0; u < 2 * DP; ++u) acc[u] = 0.f;

  const int ihi = min(i0 + BM, g.L) - 1;
  const int jlo = g.W > 0 ? max(0, i0 - g.W + 1) : 0;
  for (int t = jlo / BN; t <= ihi / BN; ++t) {
    const int j0 = t * BN;
    __syncthreads();
    load_rows<D>(Ks, k + kbase + (size_t)j0 * D, BN, min(BN, g.L - j0));
    load_rows<D>(Vs, v + kbase + (size_t)j0 * D, BN, min(BN, g.L - j0));
    __syncthreads();

    float s[CPT], dp[CPT];
#pragma unroll
    for (int mm = 0; mm < CPT; ++mm) s[mm] = dp[mm] = 0.f;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(Qs + r * LDS);
    const uint32_t* grow = reinterpret_cast<const uint32_t*>(Gs + r * LDS);
#pragma unroll 2
    for (int d2 = 0; d2 < D / 2; ++d2) {
      const float2 qa = bf2f(qrow[d2]);
      const float2 ga = bf2f(grow[d2]);
#pragma unroll
      for (int mm = 0; mm < CPT; ++mm) {
        const int jj = c + TPR * mm;
        const float2 kb = bf2f(reinterpret_cast<const uint32_t*>(Ks + jj * LDS)[d2]);
        const float2 vb = bf2f(reinterpret_cast<const uint32_t*>(Vs + jj * LDS)[d2]);
        s[mm] = fmaf(qa.x, kb.x, fmaf(qa.y, kb.y, s[mm]));
        dp[mm] = fmaf(ga.x, vb.x, fmaf(ga.y, vb.y, dp[mm]));
      }
    }
#pragma unroll
    for (int mm = 0; mm < CPT; ++mm) {
      const int jj = c + TPR * mm, j = j0 + jj;
      const bool ok = i < g.L && j < g.L && in_band(i, j, g.W);
      const float p = ok ? exp2f(fmaf(s[mm], sl2, -lse_l2)) : 0.f;
      Ss[r * (BN + 1) + jj] = p * (dp[mm] - dl);
    }
    __syncwarp();
    const float* srow = Ss + r * (BN + 1);
#pragma unroll 2
    for (int jj = 0; jj < BN; ++jj) {
      const float ds = srow[jj];
      const uint32_t* kr = reinterpret_cast<const uint32_t*>(Ks + jj * LDS);
#pragma unroll
      for (int u = 0; u < DP; ++u) {
        const float2 kb = bf2f(kr[c + TPR * u]);
        acc[2 * u] = fmaf(ds, kb.x, acc[2 * u]);
        acc[2 * u + 1] = fmaf(ds, kb.y, acc[2 * u + 1]);
      }
    }
    __syncwarp();
  }
  if (i < g.L) {
    float2* row = reinterpret_cast<float2*>(dq + qbase + (size_t)i * D);
#pragma unroll
    for (int u = 0; u < DP; ++u) row[c + TPR * u] = make_float2(acc[2 * u] * g.scale, acc[2 * u + 1] * g.scale);
  }
}

constexpr int kFwdBM = 64, kFwdBN = 32;
constexpr int kKvBN = 32, kKvBM = 32;
constexpr int kDqBM = 64, kDqBN = 32;

template <int D>
constexpr size_t fwd_smem() {
  return (size_t)(kFwdBM + 2 * kFwdBN) * (D + kPad) * 2 + (size_t)kFwdBM * (kFwdBN + 1) * 4;
}
template <int D>
constexpr size_t dkdv_smem() {
  return (size_t)(2 * kKvBN + 2 * kKvBM) * (D + kPad) * 2 + (size_t)2 * kKvBN * (kKvBM + 1) * 4 + 2 * kKvBM * 4;
}
template <int D>
constexpr size_t dq_smem() {
  return (size_t)(2 * kDqBM + 2 * kDqBN) * (D + kPad) * 2 + (size_t)kDqBM * (kDqBN + 1) * 4;
}

template <typename K>
cudaError_t prep(K kernel, size_t smem) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

template <int D>
cudaError_t fwd_d(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v, float* o, float* lse,
                  cudaStream_t s) {
  auto kern = fwd_simt_kernel<D, kFwdBM, kFwdBN>;
  constexpr size_t sm = fwd_smem<D>();
  cudaError_t e = prep(kern, sm);
  if (e != cudaSuccess) return e;
  dim3 grid((g.L + kFwdBM - 1) / kFwdBM, g.Hq, g.B);
  kern<<<grid, kThreads, sm, s>>>(g, q, k, v, o, lse);
  return cudaGetLastError();
}

template <int D>
cudaError_t dkdv_d(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dO,
                   const float* lse, const float* delta, float* dk, float* dv, cudaStream_t s) {
  auto kern = dkdv_simt_kernel<D, kKvBN, kKvBM>;
  constexpr size_t sm = dkdv_smem<D>();
  cudaError_t e = prep(kern, sm);
  if (e != cudaSuccess) return e;
  dim3 grid((g.L + kKvBN - 1) / kKvBN, g.Hkv, g.B);
  kern<<<grid, kThreads, sm, s>>>(g, q, k, v, dO, lse, delta, dk, dv);
  return cudaGetLastError();
}

template <int D>
cudaError_t dq_d(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dO,
                 const float* lse, const float* delta, float* dq, cudaStream_t s) {
  auto kern = dq_simt_kernel<D, kDqBM, kDqBN>;
  constexpr size_t sm = dq_smem<D>();
  cudaError_t e = prep(kern, sm);
  if (e != cudaSuccess) return e;
  dim3 grid((g.L + kDqBM - 1) / kDqBM, g.Hq, g.B);
  kern<<<grid, kThreads, sm, s>>>(g, q, k, v, dO, lse, delta, dq);
  return cudaGetLastError();
}

}  // namespace

#define SWA_DISPATCH_D(D_, CALL)                         \
  switch (D_) {                                          \
    case 64: return CALL(64);                            \
    case 128: return CALL(128);                          \
    case 256: return CALL(256);                          \
    case 512: return CALL(512);                          \
    default: return cudaErrorInvalidValue;               \
  }

cudaError_t launch_fwd_simt(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v, float* o,
                            float* lse, cudaStream_t s) {
#define CALL(DD) fwd_d<DD>(g, q, k, v, o, lse, s)
  SWA_DISPATCH_D(g.D, CALL)
#undef CALL
}

cudaError_t launch_delta(const Geom& g, const float* o, const uint16_t* dO, float* delta, cudaStream_t s) {
  const long rows = (long)g.B * g.Hq * g.L;
  const long blocks = (rows * 32 + kThreads - 1) / kThreads;
  delta_kernel<<<(unsigned)blocks, kThreads, 0, s>>>(rows, g.D, o, dO, delta);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv_simt(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                 const uint16_t* dO, const float* lse, const float* delta, float* dk, float* dv,
                                 cudaStream_t s) {
#define CALL(DD) dkdv_d<DD>(g, q, k, v, dO, lse, delta, dk, dv, s)
  SWA_DISPATCH_D(g.D, CALL)
#undef CALL
}

cudaError_t launch_bwd_dq_simt(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               const uint16_t* dO, const float* lse, const float* delta, float* dq,
                               cudaStream_t s) {
#define CALL(DD) dq_d<DD>(g, q, k, v, dO, lse, delta, dq, s)
  SWA_DISPATCH_D(g.D, CALL)
#undef CALL
}

}  // namespace swa
