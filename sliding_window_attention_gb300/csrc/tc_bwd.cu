// Tensor-core backward for sm_103a (head dims 64, 128, 256): a key-outer dK/dV
// pass and a query-outer dQ pass, both on tcgen05 with accumulators in Tensor
// Memory and operands staged by TMA.  P is recomputed from the forward's lse
// instead of being stored ("Training -- design (ORPO, flash-CCE head, prefix
// sharing, segmented backward)", section 6), and only tile pairs that meet
// the causal / window band are visited ("Lab 028 lab detail: Off NVIDIA, you
// fix the platform yourself", "What I changed, in plain terms" items 3-4).
//
// dK/dV, per (128-row key tile, kv head), for every query head of the group
// and every 128-row query tile in band:
//     S^T  = K Q^T,  dP^T = V dO^T                 (SS MMAs, fp32 in TMEM)
//     P^T  = exp(scale S^T - lse),  dS^T = P^T (dP^T - Delta)   (thread = key row)
//     dV  += P^T dO,  dK += dS^T Q                  (TS MMAs, A operand in TMEM)
//   dK and dV stay in TMEM for the whole group loop: no atomics, deterministic.
//   Head dim <= 128: one CTA holds both (dkdv128_tc_kernel).  Head dim 256:
//   a 2-CTA cluster, dV on one SM and dK on the other, P^T passed between
//   them through L2 (dkdv256_pair_kernel).
// dQ kernel, one CTA per (128-row query tile, query head):
//   for every key tile in band: S = Q K^T, dP = dO V^T,
//   dS = P (dP - Delta), dQ += dS K.  No read-modify-write of dQ in memory.
//
// Warp roles: warp 0 TMA producer, warp 1 TMEM owner and the single-thread
// MMA issuer, warps 2..5 and 6..9 two elementwise softmax-gradient
// warpgroups (one TMEM lane, i.e. one row, per thread), each on half of the
// columns of every step; the cluster kernel adds warps for its second
// producer and its cross-CTA traffic.
// Every mbarrier wait is bounded (see tc_ptx.cuh).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <type_traits>

#include "swa_internal.h"
#include "tc_ptx.cuh"

namespace swa {
namespace {

using namespace tc;

constexpr int kThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-5 and 6-9: two elementwise warpgroups
constexpr float kLog2e = 1.4426950408889634f;
constexpr size_t kMinSmem = 120 * 1024;  // keep one CTA per SM (each owns all 512 TMEM columns)
constexpr int kSmemMax = 232448;         // dynamic shared memory per block on sm_103 (227 KB)

// Backward preparation in one launch.  Segments 0-2 (blockIdx.y): fp16
// copies of q, k and v, four 16-byte vectors in flight per thread.  Segment 3:
// for every row of dO, its fp16 copy (scaled by the power of two s that the
// absmax pass fixed, see dscale_offset) together with the row statistics, so
// dO is read once for both; a warp per row, grid-stride.  The statistics are
// two planes of BH * Lpad floats: per (bh = b*Hq + h, i < Lpad)
// stats[bh Lpad + i] = lse_i * log2(e) and stats[BH Lpad + bh Lpad + i] =
// s * Delta_i = s * (dO_i . o_i); zero for padding rows i >= Lq.  Planar, so
// that one 16-byte load gives four columns' values.  A finite input that
// overflows fp16 latches kStatusFp16Range.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, bool& overflow, float mul = 1.f) {
  const float lo = __uint_as_float(w << 16) * mul, hi = __uint_as_float(w & 0xffff0000u) * mul;
  const __half2 hv = __floats2half2_rn(lo, hi);
  const float2 back = __half22float2(hv);
  overflow |= (isinf(back.x) && !isinf(lo)) || (isinf(back.y) && !isinf(hi));
  return *reinterpret_cast<const uint32_t*>(&hv);
}

// The dO scale s = 2^k from the largest |dO| (as a bf16 bit pattern with the
// sign cleared): the scaled maximum lands in [4, 8).  All-zero dO, or a
// non-finite maximum, keeps s = 1; k is clamped to [-125, 125] so that s and
// 1/s are normal floats.
__device__ __forceinline__ int dscale_log2(uint32_t maxbits) {
  if (maxbits == 0u || maxbits >= 0x7f80u) return 0;
  const int e = (int)(maxbits >> 7) - 127;  // floor(log2 max) (bf16 subnormals give -127)
  const int k = 2 - e;
  return k < -125 ? -125 : (k > 125 ? 125 : k);
}

// Gradient of the attention sinks (one logit c_h per query head, a term of
// every row's softmax normaliser that carries no value):
//   dc_h = - sum_{b, i} exp(c_h - lse_i) Delta_i
// over every batch and query row of head h.  c_h enters o_i only through
// lse_i, and d o_i / d c_h = -exp(c_h - lse_i) o_i; with dO_i that gives
// -exp(c_h - lse_i) Delta_i, Delta_i = dO_i . o_i.  Read from the backward's
// row statistics: lse log2 e and s Delta planes, 1/s in the scale tail.  One
// block per head; each thread sums its rows in ascending order in fp64 and a
// fixed tree combines the threads, so the result does not depend on timing.
__global__ void __launch_bounds__(256) sink_grad_kernel(const float* __restrict__ stats, int Lpad, int B, int Hq,
                                                        int Lq, const float* __restrict__ sinks,
                                                        float* __restrict__ dsinks, long long tail) {
  __shared__ double red[256];
  const int h = blockIdx.x;
  const float c2 = sinks[h] * kLog2e;
  const size_t plane = (size_t)B * Hq * Lpad;
  double acc = 0.0;
  const long long n = (long long)B * Lq;
  for (long long r = threadIdx.x; r < n; r += blockDim.x) {
    const int b = (int)(r / Lq), i = (int)(r - (long long)b * Lq);
    const size_t row = ((size_t)b * Hq + h) * Lpad + i;
    acc += (double)exp2f(c2 - stats[row]) * (double)stats[plane + row];
  }
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) dsinks[h] = (float)(-red[0] * (double)stats[tail + 1]);
}

// Per-block maxima of |dO| (bit patterns of bf16 with the sign cleared,
// which order like the magnitudes for every non-NaN value) into the stats
// tail; kAbsmaxBlocks blocks, grid-stride over 16-byte vectors.
__global__ void __launch_bounds__(256) bwd_dscale_kernel(const uint4* __restrict__ dO, long long n16,
                                                          uint32_t* __restrict__ partial,
                                                          int* __restrict__ counters) {
  if (blockIdx.x == 0 && threadIdx.x < 2) counters[threadIdx.x] = 0;  // persistent passes start at item 0
  uint32_t m = 0;
  const long long stride = (long long)gridDim.x * blockDim.x;
  long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  auto upd = [&](const uint4 a) {
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t lo = w[u] & 0x7fffu, hi = (w[u] >> 16) & 0x7fffu;
      m = max(m, max(lo, hi));
    }
  };
  for (; idx + 3 * stride < n16; idx += 4 * stride) {
    const uint4 a = __ldg(dO + idx), b = __ldg(dO + idx + stride);
    const uint4 c = __ldg(dO + idx + 2 * stride), d = __ldg(dO + idx + 3 * stride);
    upd(a);
    upd(b);
    upd(c);
    upd(d);
  }
  for (; idx < n16; idx += stride) upd(__ldg(dO + idx));
  m = __reduce_max_sync(0xffffffffu, m);
  __shared__ uint32_t wmax[8];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t b = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) b = max(b, wmax[i]);
    partial[blockIdx.x] = b;
  }
}

struct PrepParams {
  const uint16_t* src[3];
  uint16_t* dst[3];
  long long n[3];  // elements (multiples of 8)
  int BH, L, Lpad, D;  // rows of dO: BH x L (L = query rows), padded to Lpad
  const float* o;
  const uint16_t* dO;
  uint16_t* g16;
  const float* lse;
  float* stats;
  float* dscale;  // stats tail: [0] = s, [1] = 1/s, [4 ...] absmax partials
  int* status;
};

__global__ void __launch_bounds__(256) bwd_prep_kernel(const PrepParams p) {
  bool overflow = false;
  const int seg = blockIdx.y;
  if (seg < 3) {
    const uint4* src = reinterpret_cast<const uint4*>(p.src[seg]);
    uint4* dst = reinterpret_cast<uint4*>(p.dst[seg]);
    const long long n16 = p.n[seg] / 8;
    const long long stride = (long long)gridDim.x * blockDim.x;
    long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    for (; idx + 3 * stride < n16; idx += 4 * stride) {
      const uint4 a = __ldcs(src + idx), b = __ldcs(src + idx + stride);
      const uint4 c = __ldcs(src + idx + 2 * stride), d = __ldcs(src + idx + 3 * stride);
      const uint4 v4[4] = {a, b, c, d};
#pragma unroll
      for (int u = 0; u < 4; ++u)
        dst[idx + u * stride] = make_uint4(bf16x2_to_f16x2(v4[u].x, overflow), bf16x2_to_f16x2(v4[u].y, overflow),
                                           bf16x2_to_f16x2(v4[u].z, overflow), bf16x2_to_f16x2(v4[u].w, overflow));
    }
    for (; idx < n16; idx += stride) {
      const uint4 a = __ldcs(src + idx);
      dst[idx] = make_uint4(bf16x2_to_f16x2(a.x, overflow), bf16x2_to_f16x2(a.y, overflow),
                            bf16x2_to_f16x2(a.z, overflow), bf16x2_to_f16x2(a.w, overflow));
    }
  } else {
    // the dO scale from the absmax pass's per-block maxima (every block of
    // this segment reduces them; they are 1.2 KB and sit in L2)
    __shared__ uint32_t smax[8];
    const uint32_t* part = reinterpret_cast<const uint32_t*>(p.dscale + 4);
    uint32_t m = 0;
    for (int b = threadIdx.x; b < kAbsmaxBlocks; b += blockDim.x) m = max(m, part[b]);
    m = __reduce_max_sync(0xffffffffu, m);
    if ((threadIdx.x & 31) == 0) smax[threadIdx.x >> 5] = m;
    __syncthreads();
    m = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = max(m, smax[i]);
    const int kexp = dscale_log2(m);
    const float sc = __int_as_float((127 + kexp) << 23), inv_sc = __int_as_float((127 - kexp) << 23);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      p.dscale[0] = sc;
      p.dscale[1] = inv_sc;
    }
    const int lane = threadIdx.x & 31;
    const long rows = (long)p.BH * p.Lpad;
    const long nwarps = (long)gridDim.x * (blockDim.x / 32);
    for (long row = (long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; row < rows; row += nwarps) {
      const int bh = (int)(row / p.Lpad), i = (int)(row % p.Lpad);
      float acc = 0.f, l2 = 0.f;
      if (i < p.L) {
        const size_t off = ((size_t)bh * p.L + i) * p.D;
        for (int d = lane * 4; d < p.D; d += 128) {
          const float4 ov = __ldcs(reinterpret_cast<const float4*>(p.o + off + d));
          const uint2 gv = __ldcs(reinterpret_cast<const uint2*>(p.dO + off + d));
          acc = fmaf(ov.x, __uint_as_float(gv.x << 16), acc);
          acc = fmaf(ov.y, __uint_as_float(gv.x & 0xffff0000u), acc);
          acc = fmaf(ov.z, __uint_as_float(gv.y << 16), acc);
          acc = fmaf(ov.w, __uint_as_float(gv.y & 0xffff0000u), acc);
          *reinterpret_cast<uint2*>(p.g16 + off + d) =
              make_uint2(bf16x2_to_f16x2(gv.x, overflow, sc), bf16x2_to_f16x2(gv.y, overflow, sc));
        }
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sh);
        acc *= sc;  // exact: a power of two
        l2 = p.lse[(size_t)bh * p.L + i] * kLog2e;
      }
      if (lane == 0) {
        p.stats[row] = l2;
        p.stats[(size_t)p.BH * p.Lpad + row] = acc;
      }
    }
  }
  if (overflow) atomicCAS(p.status, 0, kStatusFp16Range);
}


// dQ elementwise step for one query row (lse*log2e = l2, Delta = dl) and 32
// key columns: dS = P (dP - Delta) as fp16 pairs.
// Unless FULL, key columns outside the row's visible keys v (tile-local;
// see vis(), TWO under a shared-prefix plan) get P = 0.
template <bool FULL, bool TWO = false>
__device__ __forceinline__ void dq_chunk(const uint32_t (&sv)[32], const uint32_t (&dv)[32], float sl2, float l2,
                                         float dl, int cbase, const int4& v, uint32_t (&dd)[16]) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    float p0 = fast_exp2(fmaf(__uint_as_float(sv[e]), sl2, -l2));
    float p1 = fast_exp2(fmaf(__uint_as_float(sv[e + 1]), sl2, -l2));
    if (!FULL) {
      p0 = vis<TWO>(cbase + e, v) ? p0 : 0.f;
      p1 = vis<TWO>(cbase + e + 1, v) ? p1 : 0.f;
    }
    dd[e >> 1] = pack_half2(p0 * (__uint_as_float(dv[e]) - dl), p1 * (__uint_as_float(dv[e + 1]) - dl));
  }
}


struct BwdParams {
  Geom g;
  float* out0;  // dkdv: dk ; dq: dq
  float* out1;  // dkdv: dv
  const float* stats;  // two planes: lse * log2e, then Delta (B * Hq * Lpad floats each)
  const uint16_t* x16;  // dQ at head dim 256: the fp16 copy of q (its rows go into Tensor Memory)
  int Lpad;
  int n_tiles;
  int* status;
};

// ===========================================================================
// dK / dV for head dim <= 128 with 128-row query steps, so that every MMA has
// N = 128 (tcgen05.mma with N <= 64 costs a fixed ~50 cycles per instruction
// and runs at ~60% of the tensor rate).
//
// TMEM: dV [0, 128), dK [128, 256), S^T [256, 384), dP^T [384, 512), each
// single-buffered.  Per step n the elementwise warps read S^T(n) as soon as it
// lands (the S buffer is then free for S^T(n + 1)) and compute P^T(n) while
// the tensor pipe runs dV(n - 1), dK(n - 1) and dP^T(n); once dP^T(n) has been
// read by both warpgroups they pack P^T(n) and dS^T(n) as fp16 pairs into the
// dP buffer, where dV(n) and dK(n) read them as TMEM A operands.  The
// per-column row statistics (lse, Delta) of a step are loaded into registers
// before the waits for S^T and dP^T, so their latency overlaps the MMAs; dS
// is formed from the fp16-rounded P that dV uses.  MMA issue
// order: S(n + 1) | dV(n) dK(n) | dP(n + 1); tcgen05 MMAs of one thread run in
// issue order, so dP(n + 1) overwrites the buffer only after dV(n) and dK(n)
// have read it.  Q and dO travel in separate TMA rings (Q lives from S(n) to
// dK(n), dO from dP(n) to dV(n)).
template <int D>
struct Kv128Cfg {
  static constexpr int BNK = 128, BM = 128, CW = 64;  // CW: query columns per warpgroup
  static constexpr int KCH = D / 64;
  static constexpr int KV_BYTES = BNK * D * 2;
  static constexpr int QT_BYTES = BM * D * 2;
  static constexpr int NQ = (D <= 64) ? 4 : 3;  // Q ring depth
  static constexpr int NG = (D <= 64) ? 4 : 2;  // dO ring depth
  static constexpr int DV_COL = 0, DK_COL = 128, S_COL = 256, DP_COL = 384;
  static constexpr size_t SMEM = 2 * (size_t)KV_BYTES + (size_t)(NQ + NG) * QT_BYTES + 1024 + 512;
  static_assert(SMEM <= (size_t)kSmemMax, "shared memory");
  static_assert(D <= 128, "dV and dK below the S buffer");
};

// P^T for one key row and 64 query columns (fp32, in place over S^T); lv
// holds lse * log2e of the 64 columns (loaded before S^T was waited for).
// Unless FULL, columns outside the key's visible rows v (tile-local; see
// vis(), TWO under a shared-prefix plan) get P = 0.
template <bool FULL, bool TWO = false>
__device__ __forceinline__ void kv_p64(uint32_t (&sv)[64], const float (&lv)[64], float sl2, int cbase,
                                       const int4& v) {
#pragma unroll
  for (int e = 0; e < 64; ++e) {
    float pv = fast_exp2(fmaf(__uint_as_float(sv[e]), sl2, -lv[e]));
    if (!FULL) pv = vis<TWO>(cbase + e, v) ? pv : 0.f;
    sv[e] = __float_as_uint(pv);
  }
}

// TWO: a shared-prefix plan is active (a key may be seen by two row
// intervals); a separate instantiation keeps the plain kernel's registers.
constexpr int kThreadsKv128 = 352;  // the common roles plus the dO producer (warp 10)
template <int D, bool TWO>
__global__ void __launch_bounds__(kThreadsKv128, 1)
    dkdv128_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                      const __grid_constant__ CUtensorMap tmO0,  // fp32 dk, 32 x 32 boxes
                      const __grid_constant__ CUtensorMap tmO1,  // fp32 dv
                      const BwdParams p) {
  using C = Kv128Cfg<D>;
  constexpr int BNK = C::BNK, BM = C::BM, NQ = C::NQ, NG = C::NG, KCH = C::KCH, CW = C::CW;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sK = base;
  unsigned char* sV = sK + C::KV_BYTES;
  unsigned char* sQ = sV + C::KV_BYTES;
  unsigned char* sG = sQ + NQ * C::QT_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sG + NG * C::QT_BYTES);
  uint64_t* kv_full = bars;            // [1]
  uint64_t* q_full = kv_full + 1;      // [NQ]
  uint64_t* q_empty = q_full + NQ;     // [NQ]
  uint64_t* g_full = q_empty + NQ;     // [NG]
  uint64_t* g_empty = g_full + NG;     // [NG]
  uint64_t* s_full = g_empty + NG;     // [1] S^T(n) in TMEM
  uint64_t* s_read = s_full + 1;       // [1] both warpgroups loaded S^T(n)
  uint64_t* dp_full = s_read + 1;      // [1] dP^T(n) in TMEM
  uint64_t* dp_read = dp_full + 1;     // [1] both warpgroups loaded dP^T(n)
  uint64_t* p_full = dp_read + 1;      // [1] P^T(n), dS^T(n) packed into the dP buffer
  uint64_t* acc_done = p_full + 1;     // [1]
  uint64_t* mma_drain = acc_done + 1;  // [1] every issued MMA finished (before TMEM is released)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const Geom& g = p.g;
  const int warp = threadIdx.x / 32;
  const int bkv = blockIdx.x;  // b * Hkv + kv head
  const int b = bkv / g.Hkv, kvh = bkv - b * g.Hkv;
  const int j0 = (int)blockIdx.y * BNK;
  const int jhi = min(j0 + BNK, g.L) - 1;
  // query tiles that can see a key of this tile
  const TileSteps qsteps = key_steps(g, j0, jhi, BM);
  const int ntq = qsteps.count();
  const int N = g.G * ntq;  // steps (head of group, query tile)
  if (N == 0) {
    // no query sees these keys: zero gradients (see dkdv_tc_kernel)
    zero_rows(p.out0, bkv, j0, BNK, g.L, D);
    zero_rows(p.out1, bkv, j0, BNK, g.L, D);
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < NQ; ++s) {
      mbar_init(q_full + s, 1);
      mbar_init(q_empty + s, 1);
    }
    for (int s = 0; s < NG; ++s) {
      mbar_init(g_full + s, 1);
      mbar_init(g_empty + s, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_read, 256);
    mbar_init(dp_full, 1);
    mbar_init(dp_read, 256);
    mbar_init(p_full, 256);
    mbar_init(acc_done, 1);
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto step_head = [&](int n) { return b * g.Hq + kvh * g.G + n / ntq; };
  auto step_i0 = [&](int n) { return qsteps.tile(n % ntq) * BM; };

  if (warp == 0) {
    if (elect_one()) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmG);
      mbar_arrive_expect_tx(kv_full, 2 * C::KV_BYTES);
      for (int c = 0; c < KCH; ++c) {
        tma_load_3d(sK + c * BNK * 128, &tmK, kv_full, c * 64, j0, bkv);
        tma_load_3d(sV + c * BNK * 128, &tmV, kv_full, c * 64, j0, bkv);
      }
      // Q(n), the ring refilled as soon as a slot is released
      int nq = 0;
      for (; nq < N; ++nq) {
        const int s = nq % NQ;
        if (nq >= NQ && !mbar_wait(q_empty + s, ((nq / NQ) & 1) ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(q_full + s, C::QT_BYTES);
        for (int c = 0; c < KCH; ++c)
          tma_load_3d(sQ + s * C::QT_BYTES + c * BM * 128, &tmQ, q_full + s, c * 64, step_i0(nq), step_head(nq));
      }
      if (*abort_flag) {  // unwinding: the loads in flight land before shared memory is released
        mbar_wait_drain(kv_full, 0);
        drain_ring(q_full, NQ, nq);
      }
    }
  } else if (warp == 10) {
    // dO(n) on a warp of its own, so that a wait on one ring never holds up the other
    if (elect_one()) {
      int ng = 0;
      for (; ng < N; ++ng) {
        const int s = ng % NG;
        if (ng >= NG && !mbar_wait(g_empty + s, ((ng / NG) & 1) ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(g_full + s, C::QT_BYTES);
        for (int c = 0; c < KCH; ++c)
          tma_load_3d(sG + s * C::QT_BYTES + c * BM * 128, &tmG, g_full + s, c * 64, step_i0(ng), step_head(ng));
      }
      if (*abort_flag) drain_ring(g_full, NG, ng);
    }
  } else if (warp == 1) {
    if (elect_one()) {
      const uint32_t idS = idesc_f16(BNK, BM, 0, 0, 0, 0);  // K x Q^T, V x dO^T (both K-major), N = 128
      const uint32_t idG = idesc_f16(BNK, D, 0, 0, 0, 1);   // P^T x dO, dS^T x Q (A in TMEM, B MN-major)
      const uint64_t kdk = smem_desc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t vdk = smem_desc_sw128(smem_u32(sV), 16, 1024);
      bool ok = mbar_wait(kv_full, 0, abort_flag);
      auto issue_s = [&](int n) -> bool {  // S^T(n) = K Q(n)^T
        if (!mbar_wait(q_full + n % NQ, (n / NQ) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint64_t qk = smem_desc_sw128(smem_u32(sQ + (n % NQ) * C::QT_BYTES), 16, 1024);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * 128 * 128 + (ks & 3) * 32;
          mma_ss(tmem + C::S_COL, desc_add(kdk, off), desc_add(qk, off), idS, ks > 0 ? 1u : 0u);
        }
        mma_commit(s_full);
        return true;
      };
      auto issue_dp = [&](int n) -> bool {  // dP^T(n) = V dO(n)^T
        if (!mbar_wait(g_full + n % NG, (n / NG) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint64_t gk = smem_desc_sw128(smem_u32(sG + (n % NG) * C::QT_BYTES), 16, 1024);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * 128 * 128 + (ks & 3) * 32;
          mma_ss(tmem + C::DP_COL, desc_add(vdk, off), desc_add(gk, off), idS, ks > 0 ? 1u : 0u);
        }
        mma_commit(dp_full);
        return true;
      };
      if (ok) ok = issue_s(0) && issue_dp(0);
      for (int n = 0; ok && n < N; ++n) {
        // S buffer free once both warpgroups have loaded S^T(n)
        if (!mbar_wait(s_read, n & 1, abort_flag)) { ok = false; break; }
        if (n + 1 < N && !issue_s(n + 1)) { ok = false; break; }
        if (!mbar_wait(p_full, n & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint64_t gmn = smem_desc_sw128(smem_u32(sG + (n % NG) * C::QT_BYTES), BM * 128, 1024);
        const uint64_t qmn = smem_desc_sw128(smem_u32(sQ + (n % NQ) * C::QT_BYTES), BM * 128, 1024);
#pragma unroll
        for (int ks = 0; ks < BM / 16; ++ks) {
          const uint32_t acc = (n > 0 || ks > 0) ? 1u : 0u;
          mma_ts(tmem + C::DV_COL, tmem + C::DP_COL + ks * 8, desc_add(gmn, ks * 2048), idG, acc);
          mma_ts(tmem + C::DK_COL, tmem + C::DP_COL + 64 + ks * 8, desc_add(qmn, ks * 2048), idG, acc);
        }
        mma_commit(g_empty + n % NG);
        mma_commit(q_empty + n % NQ);
        if (n + 1 < N && !issue_dp(n + 1)) { ok = false; break; }
      }
      if (ok) mma_commit(acc_done);
      // every MMA issued so far has finished before TMEM is released
      mma_commit(mma_drain);
      mbar_wait_drain(mma_drain, 0);
    }
  } else {
    // warpgroup wg (warps 2-5 / 6-9) takes query columns [64 wg, 64 wg + 64);
    // warp % 4 fixes the TMEM lane quarter, i.e. the key rows
    const int wg = (warp - 2) >> 2;
    const int r = 32 * (warp & 3) + (threadIdx.x & 31);
    const int j = j0 + r;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const float sl2 = g.scale * kLog2e;
    const int cw0 = wg * CW;
    bool ok = true;
    const size_t dplane = (size_t)g.B * g.Hq * p.Lpad;  // offset of the Delta plane
    // loop invariants of the band: the query rows that see this thread's key
    // j, and those that see every key of the tile (hoisted: recomputing them
    // per step pushed the kernel past its register budget)
    const int qlo_j = band_q_lo(g, j), qhi_j = band_q_hi(g, j);
    const int qlo_all = band_q_lo(g, jhi), qhi_all = band_q_hi(g, j0);
    constexpr bool two = TWO;  // shared-prefix plan: a key may see two row intervals
    const int4 vj = key_vis(g, j, 0);  // (plan only) both row intervals of key j
    for (int n = 0; n < N; ++n) {
      const int i0 = step_i0(n);
      const float* lse_g = p.stats + (size_t)step_head(n) * p.Lpad + i0 + cw0;
      // lse * log2e of this warpgroup's 64 query columns, loaded while S^T(n) is computed
      float lv[64];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float4 l4 = __ldg(reinterpret_cast<const float4*>(lse_g) + q);
        lv[4 * q] = l4.x;
        lv[4 * q + 1] = l4.y;
        lv[4 * q + 2] = l4.z;
        lv[4 * q + 3] = l4.w;
      }
      if (!__all_sync(0xffffffffu, mbar_wait(s_full, n & 1, abort_flag))) { ok = false; break; }
      tc_fence_after();
      uint32_t sv[64];
      tmem_ld32(tmem + lane_off + C::S_COL + cw0, *reinterpret_cast<uint32_t(*)[32]>(sv));
      tmem_ld32(tmem + lane_off + C::S_COL + cw0 + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(s_read);
      // every key of the tile seen by every query of the step: the hoisted
      // plain-band bounds, or (shared-prefix plan) the two-interval test
      const bool full = ((i0 >= qlo_all) && (i0 + BM - 1 <= qhi_all)) ||
                        (two && keys_tile_full(g, j0, jhi, i0, i0 + BM - 1));
      // query columns c of this tile that see key j: i0 + c in [qlo_j, qhi_j]
      // (and, under a plan, in its second interval)
      if (full) {
        kv_p64<true>(sv, lv, sl2, cw0, make_int4(0, 0, 0, 0));
      } else if constexpr (two) {
        bool both;
        const int4 vq = vis_in_tile(vshift(vj, i0), BM, &both);
        if (__any_sync(0xffffffffu, both)) kv_p64<false, true>(sv, lv, sl2, cw0, vq);
        else kv_p64<false>(sv, lv, sl2, cw0, vq);
      } else {
        kv_p64<false>(sv, lv, sl2, cw0, make_int4(qlo_j - i0, qhi_j - i0, 1, 0));
      }
      // P^T as fp16 pairs (the dV operand); dS below uses the same rounded P
      uint32_t pp[32];
#pragma unroll
      for (int e = 0; e < 64; e += 2) pp[e >> 1] = pack_half2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
      // Delta of the 64 columns, loaded while dP^T(n) is computed
      float dl[64];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float4 d4 = __ldg(reinterpret_cast<const float4*>(lse_g + dplane) + q);
        dl[4 * q] = d4.x;
        dl[4 * q + 1] = d4.y;
        dl[4 * q + 2] = d4.z;
        dl[4 * q + 3] = d4.w;
      }
      if (!__all_sync(0xffffffffu, mbar_wait(dp_full, n & 1, abort_flag))) { ok = false; break; }
      tc_fence_after();
      uint32_t dd[32];
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // two 32-column halves keep dP^T's registers small
        uint32_t dv[32];
        tmem_ld32(tmem + lane_off + C::DP_COL + cw0 + 32 * h, dv);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 pf = __half22float2(*reinterpret_cast<const __half2*>(&pp[16 * h + (e >> 1)]));
          dd[16 * h + (e >> 1)] = pack_half2(pf.x * (__uint_as_float(dv[e]) - dl[32 * h + e]),
                                             pf.y * (__uint_as_float(dv[e + 1]) - dl[32 * h + e + 1]));
        }
      }
      tc_fence_before();
      // the packed results land on columns the other warpgroup reads: both
      // finish reading dP^T(n) first (bounded wait, not bar.sync)
      mbar_arrive(dp_read);
      if (!__all_sync(0xffffffffu, mbar_wait(dp_read, n & 1, abort_flag))) { ok = false; break; }
      // P^T -> dP buffer columns [32 wg, 32 wg + 32), dS^T -> [64 + 32 wg, ...)
      tmem_st32(tmem + lane_off + C::DP_COL + cw0 / 2, pp);
      tmem_st32(tmem + lane_off + C::DP_COL + 64 + cw0 / 2, dd);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (ok && __all_sync(0xffffffffu, mbar_wait(acc_done, 0, abort_flag))) {
      tc_fence_after();
      // warpgroup 0 writes dK (scaled), warpgroup 1 writes dV, through TMA
      // stores staged in 16 KB per warp of the (all consumed) K, V and rings
      const uint32_t col = wg == 0 ? C::DK_COL : C::DV_COL;
      const float inv_s = p.stats[dscale_offset(g, p.Lpad) + 1];  // 1/s of the scaled dO copy
      const float mul = wg == 0 ? g.scale * inv_s : inv_s;
      tmem_rows_store_tma(wg == 0 ? &tmO0 : &tmO1, tmem + lane_off + col, 0, D, mul,
                          smem_u32(base) + (uint32_t)(warp - 2) * 16384u, j - (int)(threadIdx.x & 31), bkv,
                          (int)(threadIdx.x & 31));
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) atomicCAS(p.status, 0, kStatusTimeout);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// A operand column of K-step ks (16 query rows) in a buffer where warpgroup
// w packed its 64 columns into [64 w, 64 w + 32).
__device__ __forceinline__ uint32_t packed_col(int ks) { return (uint32_t)((ks >> 2) * 64 + (ks & 3) * 8); }

// ===========================================================================
// dK / dV for head dim 256 on 2-CTA clusters, one cluster per (128-row key
// tile, kv head).  dK and dV of a key tile need all 512 TMEM columns, so they
// live in two CTAs; here the two form a cluster and P^T is computed once:
//   rank 0 (dV):  S^T = K Q^T, P^T = exp(scale S^T - lse) (masked), dV += P^T dO,
//                 and the fp16 P^T of each step is stored to an L2 scratch;
//   rank 1 (dK):  dP^T = V dO^T, dS^T = P^T (dP^T - Delta) with P^T read back
//                 from the scratch, dK += dS^T Q.
// So the pass issues S^T, dP^T, dV and dK once (8 D per pair), and the dK CTA
// holds no K: its 64 KB go to a second Q tile, and its dP^T is double
// buffered in TMEM, so that Q(n + 1) loads and dP(n + 1) runs while the
// elementwise warps form dS(n).
// rank 0: K resident (64 KB), Q in a 4-slot ring of 16 KB slices, one dO
// tile, the P^T staging, S^T double buffered in TMEM.  rank 1:
// V resident (64 KB), two Q tiles (the MN-major B of dK), dO in a 2-slot ring
// of slices; TMEM: dK [0, 256), dP^T [256, 384) and [384, 512), where dS^T(n)
// goes back as fp16 pairs for the TS-form dK(n).
// P^T crosses between the SMs through global memory (L2): rank 0's
// elementwise threads stage their 64 columns of a key row as 16-byte chunks
// in shared memory, in a layout where a warp writes (and the matching warp of
// rank 1 later reads) 512 contiguous bytes; rank 0's store thread bulk-stores
// the 32 KB tile into a scratch slot and tells rank 1, whose relay thread
// tells rank 0 when the slot has been read (one remote arrival per step each
// way).  Two scratch slots per cluster, indexed by the SM id of rank 1: one
// CTA of this kernel fills an SM, so no two resident clusters share a slot.
constexpr int kPairScratchSms = 192;
constexpr int kPairTile = 128 * 128;  // fp16 elements of one P^T tile (32 KB)
__device__ __align__(256) uint16_t g_p256_scratch[(size_t)kPairScratchSms * 2 * kPairTile];

struct Kv256PairCfg {
  static constexpr int D = 256, BNK = 128, BM = 128, CW = 64, KCH = 4;
  static constexpr int TILE = 128 * D * 2;  // 64 KB
  static constexpr int SLICE = 128 * 128;   // 16 KB
  // rank 0: K [0, TILE), dO tile [TILE, 2 TILE), Q slices [2 TILE, 2 TILE + 4 SLICE),
  // then the 32 KB staging of P^T for the bulk store to the scratch
  static constexpr int NSL0 = 4;
  static constexpr int OFF_STG0 = 2 * TILE + NSL0 * SLICE;
  static constexpr int STG_BYTES = 128 * 128 * 2;
  // rank 1: V [0, TILE), Q tiles [TILE, 3 TILE), dO slices [3 TILE, 3 TILE + 2 SLICE)
  static constexpr int NSL1 = 2;
  static constexpr int DATA0 = OFF_STG0 + STG_BYTES;
  static constexpr int DATA1 = 3 * TILE + NSL1 * SLICE;
  static constexpr int DATA = DATA0 > DATA1 ? DATA0 : DATA1;
  static constexpr uint32_t ACC_COL = 0, BUF_COL = 256;  // S^T (rank 0) / dP^T (rank 1) buffers at 256, 384
  static constexpr size_t SMEM = (size_t)DATA + 1024 + 1024;
  static_assert(SMEM <= (size_t)kSmemMax, "shared memory");
};

struct PairBars {
  uint64_t kv_full;          // resident K (rank 0) / V (rank 1)
  uint64_t t_full[2];        // dO tile (rank 0: slot 0 only) / Q tiles (rank 1)
  uint64_t t_empty[2];
  uint64_t sl_full[6];       // slice ring: Q (rank 0) / dO (rank 1)
  uint64_t sl_empty[6];
  uint64_t s_full[2];        // rank 0: S^T(n) in TMEM buffer n & 1; rank 1: dP^T(n)
  uint64_t p_full[2];        // both warpgroups packed P^T (rank 0) / dS^T (rank 1) into buffer n & 1
  uint64_t x_done[2];        // rank 0: threads stored P^T(n) to the scratch; rank 1: threads consumed it
  uint64_t x_peer[2];        // rank 0: rank 1 consumed slot n & 1; rank 1: rank 0 stored into slot n & 1
  uint64_t stg_free;         // rank 0: the bulk store has read the staging
  uint64_t acc_done, mma_drain;
  uint32_t tmem_slot;
  int abort_flag;
  int smid;                  // SM id of this CTA (rank 1's indexes the scratch)
};

// Warps: 0 TMA of the resident operand and the whole tiles, 11 TMA of the
// slices, 1 Tensor Memory owner and MMA issuer, 2-9 elementwise, 10 the
// cross-CTA traffic (rank 0: P^T bulk stores; rank 1: the relay).  Every
// thread that spins on a barrier has a warp of its own: lanes of one warp
// that spin on different barriers delay each other.
constexpr int kPairThreads = 384;
template <bool TWO>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    dkdv256_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                        const __grid_constant__ CUtensorMap tmO0,  // fp32 dk, 32 x 32 boxes
                        const __grid_constant__ CUtensorMap tmO1,  // fp32 dv
                        const BwdParams p) {
  using C = Kv256PairCfg;
  constexpr int BNK = C::BNK, BM = C::BM, CW = C::CW, KCH = C::KCH, D = C::D;
  constexpr uint32_t R = 2;  // CTAs per cluster
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PairBars* bars = reinterpret_cast<PairBars*>(base + C::DATA);
  volatile int* abort_flag = &bars->abort_flag;
  const uint32_t rank = cluster_rank();
  const bool dvr = rank == 0;  // the dV CTA (P^T producer)
  const int NSL = dvr ? C::NSL0 : C::NSL1;
  unsigned char* sRes = base;                                       // K (rank 0) / V (rank 1)
  unsigned char* sT = base + C::TILE;                               // dO tile (rank 0) / Q tiles (rank 1)
  unsigned char* sSl = base + (dvr ? 2 * C::TILE : 3 * C::TILE);    // slice ring
  unsigned char* sStg = base + C::OFF_STG0;                         // rank 0: P^T staging

  const Geom& g = p.g;
  const int warp = threadIdx.x / 32;
  const int bkv = blockIdx.x / 2;  // b * Hkv + kv head
  const int b = bkv / g.Hkv, kvh = bkv - b * g.Hkv;
  const int j0 = (int)blockIdx.y * BNK;
  const int jhi = min(j0 + BNK, g.L) - 1;
  const TileSteps qsteps = key_steps(g, j0, jhi, BM);
  const int ntq = qsteps.count();
  const int N = g.G * ntq;  // steps (head of group, query tile)
  if (N == 0) {
    // no query sees these keys: zero gradients ("Lab 028 lab detail", "What I
    // changed, in plain terms" item 5(b)); both CTAs of the cluster leave here
    // together, before any cluster barrier
    zero_rows(dvr ? p.out1 : p.out0, bkv, j0, BNK, g.L, D);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->t_full[s], 1);
      mbar_init(&bars->t_empty[s], 1);
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->p_full[s], 256);
      mbar_init(&bars->x_done[s], 256);
      mbar_init(&bars->x_peer[s], 1);
    }
    mbar_init(&bars->stg_free, 1);
    for (int s = 0; s < 6; ++s) {
      mbar_init(&bars->sl_full[s], 1);
      mbar_init(&bars->sl_empty[s], 1);
    }
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->mma_drain, 1);
    bars->abort_flag = 0;
    uint32_t sm;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
    bars->smid = sm < (uint32_t)kPairScratchSms ? (int)sm : -1;
    if (bars->smid < 0) atomicCAS(p.status, 0, kStatusScratch);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  // the scratch slots of this cluster: rank 1's SM id
  int sm1;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(sm1) : "r"(mapa(smem_u32(&bars->smid), 1u)) : "memory");
  if (sm1 < 0 && threadIdx.x == 0) cluster_abort(abort_flag, R);
  uint4* scratch = reinterpret_cast<uint4*>(g_p256_scratch + (size_t)(sm1 < 0 ? 0 : sm1) * 2 * kPairTile);
  auto step_head = [&](int n) { return b * g.Hq + kvh * g.G + n / ntq; };
  auto step_i0 = [&](int n) { return (TWO ? qsteps.tile(n % ntq) : qsteps.lo0 + n % ntq) * BM; };

  if (warp == 0) {
    const int lane = threadIdx.x & 31;
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA: resident operand, whole tiles
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmG);
      mbar_arrive_expect_tx(&bars->kv_full, C::TILE);
      for (int c = 0; c < KCH; ++c) tma_load_3d(sRes + c * C::SLICE, dvr ? &tmK : &tmV, &bars->kv_full, c * 64, j0, bkv);
      // rank 0: one dO tile buffer; rank 1: two Q tile buffers
      const int NT = dvr ? 1 : 2;
      const CUtensorMap* mt = dvr ? &tmG : &tmQ;
      int nt = 0;
      for (; nt < N; ++nt) {
        const int tb = nt % NT;
        if (nt >= NT && !mbar_wait_cl(&bars->t_empty[tb], ((nt / NT) - 1) & 1, abort_flag, R)) break;
        mbar_arrive_expect_tx(&bars->t_full[tb], C::TILE);
        for (int c = 0; c < KCH; ++c)
          tma_load_3d(sT + tb * C::TILE + c * C::SLICE, mt, &bars->t_full[tb], c * 64, step_i0(nt), step_head(nt));
      }
      if (*abort_flag) {  // unwinding: the loads in flight land before shared memory is released
        mbar_wait_drain(&bars->kv_full, 0);
        for (int k = nt - 1; k >= 0 && k >= nt - NT; --k) mbar_wait_drain(&bars->t_full[k % NT], (k / NT) & 1);
      }
    }
  } else if (warp == 11) {
    if ((threadIdx.x & 31) == 0) {
      // ---------------------------------------------------------------- TMA: 64-column slices
      const CUtensorMap* msl = dvr ? &tmQ : &tmG;
      int ns = 0;
      bool ok = true;
      for (int m = 0; ok && m < N; ++m) {
        for (int c = 0; c < KCH; ++c, ++ns) {
          const int s = ns % NSL;
          if (ns >= NSL && !mbar_wait_cl(&bars->sl_empty[s], ((ns / NSL) & 1) ^ 1, abort_flag, R)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->sl_full[s], C::SLICE);
          tma_load_3d(sSl + s * C::SLICE, msl, &bars->sl_full[s], c * 64, step_i0(m), step_head(m));
        }
      }
      if (*abort_flag) drain_ring(bars->sl_full, NSL, ns);
    }
  } else if (warp == 10) {
    const int lane = threadIdx.x & 31;
    if (lane == 0 && dvr) {
      // ---------------------------------------------------------------- P^T tiles to the scratch (rank 0)
      // once the warps staged P^T(n) and rank 1 has read what step n - 2 left
      // in slot n & 1: bulk store, staging free again once read out, rank 1
      // told once the writes are complete
      for (int n = 0; n < N; ++n) {
        const int s = n & 1;
        if (!mbar_wait_cl(&bars->x_done[s], (n >> 1) & 1, abort_flag, R)) break;
        if (n >= 2 && !mbar_wait_cl(&bars->x_peer[s], ((n >> 1) - 1) & 1, abort_flag, R)) break;
        fence_proxy_async_global();
        if (sm1 >= 0) bulk_store_s2g(scratch + (size_t)s * (kPairTile / 8), smem_u32(sStg), C::STG_BYTES);
        bulk_commit_group();
        bulk_wait_read_all();
        mbar_arrive(&bars->stg_free);
        bulk_wait_all();
        fence_proxy_async_global();
        mbar_arrive_remote(mapa(smem_u32(&bars->x_peer[s]), 1u));
      }
      bulk_wait_all();  // no store still reads this CTA's shared memory
    } else if (lane == 0) {
      // ---------------------------------------------------------------- relay (rank 1)
      // "slot n & 1 was read" -> rank 0
      for (int n = 0; n < N; ++n) {
        if (!mbar_wait_cl(&bars->x_done[n & 1], (n >> 1) & 1, abort_flag, R)) break;
        mbar_arrive_remote(mapa(smem_u32(&bars->x_peer[n & 1]), 0u));
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (elect_one()) {
      const uint32_t idS = idesc_f16(BNK, BM, 0, 0, 0, 0);  // K x Q^T, V x dO^T (both K-major), N = 128
      const uint32_t idG = idesc_f16(BNK, D, 0, 0, 0, 1);   // P^T x dO, dS^T x Q (A in TMEM, B MN-major), N = 256
      const uint64_t rdk = smem_desc_sw128(smem_u32(sRes), 16, 1024);
      bool ok = mbar_wait_cl(&bars->kv_full, 0, abort_flag, R);
      int used = 0;  // slices consumed
      // S^T (rank 0) or dP^T (rank 1): resident A, B from the slice ring, into TMEM column col
      auto issue_sliced = [&](uint32_t col) -> bool {
        for (int c = 0; c < KCH; ++c, ++used) {
          const int s = used % NSL;
          if (!mbar_wait_cl(&bars->sl_full[s], (used / NSL) & 1, abort_flag, R)) return false;
          tc_fence_after();
          const uint64_t bd = smem_desc_sw128(smem_u32(sSl + s * C::SLICE), 16, 1024);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ss(tmem + col, desc_add(rdk, c * C::SLICE + ks * 32), desc_add(bd, ks * 32), idS, (c | ks) ? 1u : 0u);
          mma_commit(&bars->sl_empty[s]);
        }
        return true;
      };
      // dV(n) / dK(n): accumulator += packed TMEM operand (buffer col) x tile tb (MN-major)
      auto issue_grad = [&](int n, uint32_t col, int tb) {
        const uint64_t tmn = smem_desc_sw128(smem_u32(sT + tb * C::TILE), BM * 128, 1024);
#pragma unroll
        for (int ks = 0; ks < BM / 16; ++ks)
          mma_ts(tmem + C::ACC_COL, tmem + col + packed_col(ks), desc_add(tmn, ks * 2048), idG,
                 (n > 0 || ks > 0) ? 1u : 0u);
        mma_commit(&bars->t_empty[tb]);
      };
      // S^T(0), S^T(1) (rank 0) or dP^T(0), dP^T(1) (rank 1) into the two buffers
      if (ok) ok = issue_sliced(C::BUF_COL);
      if (ok) mma_commit(&bars->s_full[0]);
      if (ok && N > 1) ok = issue_sliced(C::BUF_COL + 128);
      if (ok && N > 1) mma_commit(&bars->s_full[1]);
      for (int n = 0; ok && n < N; ++n) {
        const uint32_t sb = C::BUF_COL + 128 * (n & 1);
        const int tb = dvr ? 0 : (n & 1);
        const uint32_t tpar = dvr ? (n & 1) : ((n >> 1) & 1);
        if (!mbar_wait_cl(&bars->p_full[n & 1], (n >> 1) & 1, abort_flag, R) ||
            !mbar_wait_cl(&bars->t_full[tb], tpar, abort_flag, R)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_grad(n, sb, tb);  // dV(n) / dK(n); the next product into this buffer follows it in issue order
        if (n + 2 < N) {
          if (!issue_sliced(sb)) {
            ok = false;
            break;
          }
          mma_commit(&bars->s_full[n & 1]);
        }
      }
      if (ok) mma_commit(&bars->acc_done);
      // every MMA issued so far has finished before TMEM is released
      mma_commit(&bars->mma_drain);
      mbar_wait_drain(&bars->mma_drain, 0);
    }
  } else {
    // ---------------------------------------------------------------- elementwise
    // warpgroup wg (warps 2-5 / 6-9) takes query columns [64 wg, 64 wg + 64);
    // warp % 4 fixes the TMEM lane quarter, i.e. the key rows
    const int wg = (warp - 2) >> 2;
    const int r = 32 * (warp & 3) + (threadIdx.x & 31);
    const int j = j0 + r;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const float sl2 = g.scale * kLog2e;
    const int cw0 = wg * CW;
    const bool scratch_ok = sm1 >= 0;
    bool ok = true;
    const size_t dplane = (size_t)g.B * g.Hq * p.Lpad;  // offset of the Delta plane
    // rank 0: the query rows that see this thread's key j, and those that see
    // every key of the tile (hoisted out of the step loop)
    const int qlo_j = band_q_lo(g, j), qhi_j = band_q_hi(g, j);
    const int qlo_all = band_q_lo(g, jhi), qhi_all = band_q_hi(g, j0);
    constexpr bool two = TWO;  // shared-prefix plan: a key may see two row intervals
    const int4 vj = key_vis(g, j, 0);
    // 16-byte chunk k of this thread's 64 columns in a scratch slot
    // (chunk-major: a warp's 32 rows of one chunk are 512 contiguous bytes)
    const int chunk0 = (cw0 / 8) * 128 + r;
    for (int n = 0; n < N; ++n) {
      const int i0 = step_i0(n);
      const int sbuf = n & 1;
      const uint32_t scol = C::BUF_COL + 128 * sbuf;
      const float* lse_g = p.stats + (size_t)step_head(n) * p.Lpad + i0 + cw0;
      uint4* slot = scratch + (size_t)sbuf * (kPairTile / 8);
      uint32_t pp[32];  // P^T of this key row and 64 query columns, fp16 pairs
      if (dvr) {
        // lse * log2e of this warpgroup's 64 query columns, loaded while S^T(n) is computed
        float lv[64];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const float4 l4 = __ldg(reinterpret_cast<const float4*>(lse_g) + q);
          lv[4 * q] = l4.x;
          lv[4 * q + 1] = l4.y;
          lv[4 * q + 2] = l4.z;
          lv[4 * q + 3] = l4.w;
        }
        if (!__all_sync(0xffffffffu, mbar_wait_cl(&bars->s_full[sbuf], (n >> 1) & 1, abort_flag, R))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sv[64];
        tmem_ld32(tmem + lane_off + scol + cw0, *reinterpret_cast<uint32_t(*)[32]>(sv));
        tmem_ld32(tmem + lane_off + scol + cw0 + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
        tmem_wait_ld();
        const bool full = ((i0 >= qlo_all) && (i0 + BM - 1 <= qhi_all)) ||
                          (two && keys_tile_full(g, j0, jhi, i0, i0 + BM - 1));
        if (full) {
          kv_p64<true>(sv, lv, sl2, cw0, make_int4(0, 0, 0, 0));
        } else if constexpr (two) {
          bool both;
          const int4 vq = vis_in_tile(vshift(vj, i0), BM, &both);
          if (__any_sync(0xffffffffu, both)) kv_p64<false, true>(sv, lv, sl2, cw0, vq);
          else kv_p64<false>(sv, lv, sl2, cw0, vq);
        } else {
          kv_p64<false>(sv, lv, sl2, cw0, make_int4(qlo_j - i0, qhi_j - i0, 1, 0));
        }
#pragma unroll
        for (int e = 0; e < 64; e += 2) pp[e >> 1] = pack_half2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
        // the dV operand: into the first half of this warpgroup's own columns of the S buffer
        tmem_st32(tmem + lane_off + scol + cw0, pp);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full[sbuf]);
        // P^T(n) for the dK CTA: into the staging once the store of step n - 1 has read it
        if (n >= 1 && !__all_sync(0xffffffffu, mbar_wait_cl(&bars->stg_free, (n - 1) & 1, abort_flag, R))) {
          ok = false;
          break;
        }
        {
          const uint32_t st = smem_u32(sStg) + (uint32_t)chunk0 * 16u;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            st_smem_v4(st + k * 128 * 16, pp[4 * k], pp[4 * k + 1], pp[4 * k + 2], pp[4 * k + 3]);
        }
        fence_proxy_async_smem();  // the bulk store (async proxy) reads what these stores wrote
        mbar_arrive(&bars->x_done[sbuf]);
      } else {
        // Delta of the 64 columns, loaded while P^T(n) and dP^T(n) are on their way
        float dl[64];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const float4 d4 = __ldg(reinterpret_cast<const float4*>(lse_g + dplane) + q);
          dl[4 * q] = d4.x;
          dl[4 * q + 1] = d4.y;
          dl[4 * q + 2] = d4.z;
          dl[4 * q + 3] = d4.w;
        }
        if (!__all_sync(0xffffffffu, mbar_wait_cl(&bars->x_peer[sbuf], (n >> 1) & 1, abort_flag, R))) {
          ok = false;
          break;
        }
        if (scratch_ok) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {  // L2, not L1: the slot is rewritten every other step
            const uint4 w = __ldcg(slot + chunk0 + k * 128);
            pp[4 * k] = w.x;
            pp[4 * k + 1] = w.y;
            pp[4 * k + 2] = w.z;
            pp[4 * k + 3] = w.w;
          }
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) pp[k] = 0u;
        }
        if (!__all_sync(0xffffffffu, mbar_wait_cl(&bars->s_full[sbuf], (n >> 1) & 1, abort_flag, R))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t dd[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // two 32-column halves keep dP^T's registers small
          uint32_t dv[32];
          tmem_ld32(tmem + lane_off + scol + cw0 + 32 * h, dv);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 pf = __half22float2(*reinterpret_cast<const __half2*>(&pp[16 * h + (e >> 1)]));
            dd[16 * h + (e >> 1)] = pack_half2(pf.x * (__uint_as_float(dv[e]) - dl[32 * h + e]),
                                               pf.y * (__uint_as_float(dv[e + 1]) - dl[32 * h + e + 1]));
          }
        }
        // dS^T: into the first half of this warpgroup's own columns of the dP buffer
        tmem_st32(tmem + lane_off + scol + cw0, dd);
        mbar_arrive(&bars->x_done[sbuf]);  // P^T(n) consumed: the slot may be rewritten
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full[sbuf]);
      }
    }
    if (ok && __all_sync(0xffffffffu, mbar_wait_cl(&bars->acc_done, 0, abort_flag, R))) {
      tc_fence_after();
      // each warpgroup writes half of the accumulator's columns (dK scaled),
      // through TMA stores staged in 16 KB per warp of the first 128 KB (the
      // consumed resident operand and tiles; rank 0's P^T staging lies above)
      const float inv_s = p.stats[dscale_offset(g, p.Lpad) + 1];  // 1/s of the scaled dO copy
      const float mul = dvr ? inv_s : g.scale * inv_s;
      tmem_rows_store_tma(dvr ? &tmO1 : &tmO0, tmem + lane_off + C::ACC_COL + wg * (D / 2), wg * (D / 2), D / 2, mul,
                          smem_u32(base) + (uint32_t)(warp - 2) * 16384u, j - (int)(threadIdx.x & 31), bkv,
                          (int)(threadIdx.x & 31));
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) atomicCAS(p.status, 0, kStatusTimeout);
  cluster_sync();  // no CTA leaves while its peer may still arrive on its barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ===========================================================================
// dQ for head dim 256 with 64-row key steps.  Q of the CTA's 128 rows sits in
// Tensor Memory as fp16 pairs and is the A operand of S = Q K^T (TS form), so
// shared memory holds only dO (64 KB) and two stages of K and V (32 KB each):
// with Q and dO both in shared memory only 32-row key steps fit, and an MMA
// of N = 32 runs at about 29% of the tensor rate, against about 60% for
// N = 64.
// TMEM: dQ [0, 256), Q [256, 384), S [384, 448), dP and then dS [448, 512).
// Both elementwise warpgroups take every step, 32 of its 64 key columns
// each.  dS (fp16 pairs) goes back over dP, the A operand of dQ += dS K, once
// both warpgroups have read dP; dP(n + 1) is issued after dQ(n), and S(n + 1)
// as soon as S(n) and dP(n) are read.
template <int D>
struct DqCfg {
  static constexpr int BMQ = 128;  // query rows per CTA (MMA M)
  static constexpr int BN = 64;    // key rows per step (MMA N of S and dP)
  static constexpr int CW = 32;    // key columns per warpgroup
  static constexpr int KCH = D / 64;
  static constexpr int QT_BYTES = BMQ * D * 2;  // dO tile
  static constexpr int KV_BYTES = BN * D * 2;   // K or V tile (one 4-D TMA instruction)
  static constexpr int NS = 2;                  // K / V stages
  static constexpr uint32_t DQ_COL = 0, Q_COL = 256, S_COL = 384, DP_COL = 448;
  static constexpr size_t SMEM_USED = (size_t)QT_BYTES + 2 * (size_t)NS * KV_BYTES + 1024 + 1024;
  static constexpr size_t SMEM = SMEM_USED > kMinSmem ? SMEM_USED : kMinSmem;
  static_assert(SMEM <= (size_t)kSmemMax, "shared memory");
  static_assert(D == 256, "head dim 256 only (dQ fills the columns below Q, S and dP)");
};

// TWO: a shared-prefix plan is active (a row may see two key intervals); a
// separate instantiation keeps the plain kernel's code.
template <int D, bool TWO>
__global__ void __launch_bounds__(kThreads, 1)
    dq_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmG,
                 const __grid_constant__ CUtensorMap tmO,  // fp32 dq, 32 x 32 boxes
                 const BwdParams p) {
  using C = DqCfg<D>;
  constexpr int BMQ = C::BMQ, BN = C::BN, NS = C::NS, KCH = C::KCH, CW = C::CW;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sG = base;
  unsigned char* sK = sG + C::QT_BYTES;
  unsigned char* sV = sK + NS * C::KV_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + NS * C::KV_BYTES);
  uint64_t* g_full = bars;              // [1] dO landed
  uint64_t* kv_full = g_full + 1;       // [NS] K and V of a stage landed
  uint64_t* kv_empty = kv_full + NS;    // [NS] dQ of the stage's step finished (S and dP before it)
  uint64_t* q_ready = kv_empty + NS;    // [1] the elementwise threads wrote Q into Tensor Memory
  uint64_t* sdp_full = q_ready + 1;     // [1] S and dP of a step in Tensor Memory
  uint64_t* sdp_read = sdp_full + 1;    // [1] every elementwise thread read S and dP of the step
  uint64_t* ds_full = sdp_read + 1;     // [1] dS of the step written over dP
  uint64_t* acc_done = ds_full + 1;     // [1]
  uint64_t* mma_drain = acc_done + 1;   // [1] every issued MMA finished (before TMEM is released)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const Geom& g = p.g;
  const int warp = threadIdx.x / 32;
  const int bh = blockIdx.x;
  const int b = bh / g.Hq, h = bh - b * g.Hq;
  const int bkv = b * g.Hkv + h / g.G;
  const int qt = p.n_tiles - 1 - (int)blockIdx.y;  // longest rows first
  const int i0 = qt * BMQ;
  const int ihi = min(i0 + BMQ, g.Lq) - 1;
  // key tiles meeting the band of rows i0 .. ihi (never empty)
  const TileSteps ksteps = row_steps(g, i0, ihi, BN);
  const int nt = ksteps.count();
  constexpr bool two = TWO;  // shared-prefix plan: a row may see two key intervals

  if (threadIdx.x == 0) {
    mbar_init(g_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(kv_full + s, 1);
      mbar_init(kv_empty + s, 1);
    }
    mbar_init(q_ready, 256);
    mbar_init(sdp_full, 1);
    mbar_init(sdp_read, 256);
    mbar_init(ds_full, 256);
    mbar_init(acc_done, 1);
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (elect_one()) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmG);
      mbar_arrive_expect_tx(g_full, C::QT_BYTES);
      for (int c = 0; c < KCH; ++c) tma_load_3d(sG + c * BMQ * 128, &tmG, g_full, c * 64, i0, bh);
      int issued = 0;
      for (int n = 0; n < nt; ++n) {
        const int st = n % NS;
        const int j0 = (two ? ksteps.tile(n) : ksteps.lo0 + n) * BN;
        if (n >= NS && !mbar_wait(kv_empty + st, ((n / NS) & 1) ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(kv_full + st, 2 * C::KV_BYTES);
        // all KCH 64-column chunks of the BN rows in one instruction each
        tma_load_4d(sK + st * C::KV_BYTES, &tmK, kv_full + st, 0, j0, 0, bkv);
        tma_load_4d(sV + st * C::KV_BYTES, &tmV, kv_full + st, 0, j0, 0, bkv);
        ++issued;
      }
      if (*abort_flag) {  // unwinding: the loads in flight land before shared memory is released
        mbar_wait_drain(g_full, 0);
        drain_ring(kv_full, NS, issued);
      }
    }
  } else if (warp == 1) {
    if (elect_one()) {
      const uint32_t idS = idesc_f16(BMQ, BN, 0, 0, 0, 0);  // Q x K^T (Q from TMEM), dO x V^T
      const uint32_t idQ = idesc_f16(BMQ, D, 0, 0, 0, 1);   // dS x K (dS from TMEM, K MN-major)
      const uint64_t gdk = smem_desc_sw128(smem_u32(sG), 16, 1024);  // dO, K-major (resident)
      bool ok = mbar_wait(g_full, 0, abort_flag) && mbar_wait(q_ready, 0, abort_flag);
      auto issue_dq = [&](int m) -> bool {
        const int st = m % NS;
        if (!mbar_wait(ds_full, m & 1, abort_flag)) return false;
        tc_fence_after();
        const uint64_t kmn = smem_desc_sw128(smem_u32(sK + st * C::KV_BYTES), BN * 128, 1024);  // K, MN-major
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks)
          mma_ts(tmem + C::DQ_COL, tmem + C::DP_COL + ks * 8, desc_add(kmn, ks * 2048), idQ,
                 (m > 0 || ks > 0) ? 1u : 0u);
        mma_commit(kv_empty + st);
        return true;
      };
      for (int n = 0; ok && n < nt; ++n) {
        const int st = n % NS;
        if (!mbar_wait(kv_full + st, (n / NS) & 1, abort_flag)) { ok = false; break; }
        // S(n) overwrites S(n - 1): every elementwise thread has read it
        if (n >= 1 && !mbar_wait(sdp_read, (n - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint64_t kk = smem_desc_sw128(smem_u32(sK + st * C::KV_BYTES), 16, 1024);  // K, K-major
        const uint64_t vk = smem_desc_sw128(smem_u32(sV + st * C::KV_BYTES), 16, 1024);  // V, K-major
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks & 3) * 32, ck = (ks >> 2) * BN * 128;
          mma_ts(tmem + C::S_COL, tmem + C::Q_COL + ks * 8, desc_add(kk, ck + off), idS, ks > 0 ? 1u : 0u);
        }
        // dP(n) overwrites dS(n - 1), which dQ(n - 1) reads: issue that first
        if (n >= 1 && !issue_dq(n - 1)) { ok = false; break; }
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks & 3) * 32, cq = (ks >> 2) * BMQ * 128, ck = (ks >> 2) * BN * 128;
          mma_ss(tmem + C::DP_COL, desc_add(gdk, cq + off), desc_add(vk, ck + off), idS, ks > 0 ? 1u : 0u);
        }
        mma_commit(sdp_full);
      }
      if (ok && issue_dq(nt - 1)) mma_commit(acc_done);
      // every MMA issued so far has finished before TMEM is released
      mma_commit(mma_drain);
      mbar_wait_drain(mma_drain, 0);
    }
  } else {
    const int wg = (warp - 2) >> 2;  // warps 2-5 / 6-9, see the dK/dV kernel
    const int r = 32 * (warp & 3) + (threadIdx.x & 31);
    const int i = i0 + r;
    const bool row_ok = i < g.Lq;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const float sl2 = g.scale * kLog2e;
    {
      // Q row i into Tensor Memory as fp16 pairs (one 32-bit column per two
      // head-dim elements): warpgroup wg fills columns [64 wg, 64 wg + 64) of
      // Q, head-dim elements [128 wg, 128 wg + 128)
      const uint4* src = reinterpret_cast<const uint4*>(p.x16 + ((size_t)bh * g.Lq + (row_ok ? i : 0)) * D) + wg * 16;
#pragma unroll 1
      for (int j = 0; j < 2; ++j) {
        uint32_t v[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 w4 = row_ok ? __ldg(src + j * 8 + q) : make_uint4(0u, 0u, 0u, 0u);
          v[4 * q] = w4.x;
          v[4 * q + 1] = w4.y;
          v[4 * q + 2] = w4.z;
          v[4 * q + 3] = w4.w;
        }
        tmem_st32(tmem + lane_off + C::Q_COL + wg * 64 + j * 32, v);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(q_ready);
    }
    const float2 rs = row_ok ? make_float2(p.stats[(size_t)bh * p.Lpad + i],
                                           p.stats[((size_t)g.B * g.Hq + bh) * p.Lpad + i])
                             : make_float2(0.f, 0.f);
    // key columns of this warpgroup: cb0 .. cb0 + CW - 1 of each step
    const int cb0 = wg * CW;
    bool ok = true;
    // loop invariants: this row's band, and the bounds every row of the tile shares
    const int4 vrow = row_vis(g, i, 0);
    const int lo_all = band_key_lo(g, ihi), hi_all = band_key_hi(g, i0);
    for (int n = 0; n < nt; ++n) {
      const int j0 = (two ? ksteps.tile(n) : ksteps.lo0 + n) * BN;
      if (!__all_sync(0xffffffffu, mbar_wait(sdp_full, n & 1, abort_flag))) { ok = false; break; }
      tc_fence_after();
      uint32_t sv[CW], dv[CW];
      tmem_ld32(tmem + lane_off + C::S_COL + cb0, sv);
      tmem_ld32(tmem + lane_off + C::DP_COL + cb0, dv);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(sdp_read);  // S may be overwritten; dP once both warpgroups have read it
      const bool full = two ? rows_tile_full(g, i0, ihi, j0, j0 + BN - 1) : (j0 >= lo_all && j0 + BN - 1 <= hi_all);
      // key columns c of this tile visible to row i: j0 + c in the row's band
      bool both = false;
      const int4 vv = two ? vis_in_tile(vshift(vrow, j0), BN, &both) : vshift(vrow, j0);
      const bool two_here = two && __any_sync(0xffffffffu, both);
      uint32_t dd[CW / 2];
      if (full) dq_chunk<true>(sv, dv, sl2, rs.x, rs.y, cb0, vv, dd);
      else if (two_here) dq_chunk<false, true>(sv, dv, sl2, rs.x, rs.y, cb0, vv, dd);
      else dq_chunk<false>(sv, dv, sl2, rs.x, rs.y, cb0, vv, dd);
      // dS of keys cb0 .. cb0 + 31 goes to columns cb0 / 2 .. of the dP
      // buffer, which the other warpgroup may still be reading
      if (!__all_sync(0xffffffffu, mbar_wait(sdp_read, n & 1, abort_flag))) { ok = false; break; }
      tc_fence_after();
      tmem_st16(tmem + lane_off + C::DP_COL + cb0 / 2, dd);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(ds_full);
    }
    if (ok && __all_sync(0xffffffffu, mbar_wait(acc_done, 0, abort_flag))) {
      tc_fence_after();
      // each warpgroup writes half of the dQ columns, through TMA stores
      // staged in 16 KB per warp of the (all consumed) tiles and rings
      const float mul = g.scale * p.stats[dscale_offset(g, p.Lpad) + 1];  // scale / s
      tmem_rows_store_tma(&tmO, tmem + lane_off + C::DQ_COL + wg * (D / 2), wg * (D / 2), D / 2, mul,
                          smem_u32(base) + (uint32_t)(warp - 2) * 16384u, i - (int)(threadIdx.x & 31), bh,
                          (int)(threadIdx.x & 31));
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) atomicCAS(p.status, 0, kStatusTimeout);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ===========================================================================
// dQ for head dim <= 128 with 128-row key steps, so every MMA has N >= 128
// (tcgen05.mma with N <= 64 costs a fixed ~50 cycles per instruction and runs
// at ~60% of the tensor rate; N >= 128 runs at the full rate).
//
// TMEM: dQ [0, D), two S buffers [128, 256) and [256, 384), one dP buffer
// [384, 512).  Each warpgroup handles 64 of the 128 key columns of a step.
// dS (fp16 pairs) is written back over the S buffer it came from, so the dP
// buffer is free as soon as both warpgroups have read it: dP(n+1) is issued
// while step n's elementwise work is still running.  S(n+2) reuses S(n)'s
// buffer and is issued right after dQ(n), which reads dS(n) from it.
// K tiles (used by S(n) and dQ(n)) and V tiles (used only by dP(n)) travel in
// separate TMA rings so a V tile is released early.
template <int D>
struct Dq128Cfg {
  static constexpr int BMQ = 128, BN = 128, CW = 64;  // CW: key columns per warpgroup
  static constexpr int KCH = D / 64;
  static constexpr int QT_BYTES = BMQ * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int NK = (D <= 64) ? 4 : 3;   // K ring depth
  static constexpr int NV = (D <= 64) ? 4 : 2;   // V ring depth
  static constexpr int DQ_COL = 0, S_COL = 128, DP_COL = 384;
  static constexpr size_t SMEM = 2 * (size_t)QT_BYTES + (size_t)(NK + NV) * KV_BYTES + 1024 + 1024;
  static_assert(SMEM <= (size_t)kSmemMax, "shared memory");
  static_assert(D <= 128, "dQ below the S buffers");
};

// TWO: a shared-prefix plan is active (a row may see two key intervals); a
// separate instantiation keeps the plain kernel's code.
template <int D, bool TWO>
__global__ void __launch_bounds__(kThreadsKv128, 1)
    dq128_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                    const __grid_constant__ CUtensorMap tmO,  // fp32 dq, 32 x 32 boxes
                    const BwdParams p) {
  using C = Dq128Cfg<D>;
  constexpr int BMQ = C::BMQ, BN = C::BN, NK = C::NK, NV = C::NV, KCH = C::KCH, CW = C::CW;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sQ = base;
  unsigned char* sG = sQ + C::QT_BYTES;
  unsigned char* sK = sG + C::QT_BYTES;
  unsigned char* sV = sK + NK * C::KV_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + NV * C::KV_BYTES);
  uint64_t* q_full = bars;              // [1]
  uint64_t* k_full = q_full + 1;        // [NK]
  uint64_t* k_empty = k_full + NK;      // [NK]
  uint64_t* v_full = k_empty + NK;      // [NV]
  uint64_t* v_empty = v_full + NV;      // [NV]
  uint64_t* sdp_full = v_empty + NV;    // [2] S(n) and dP(n) of step n are in TMEM
  uint64_t* ds_full = sdp_full + 2;     // [2] dS(n) written over S buffer n % 2
  uint64_t* ldd = ds_full + 2;          // [2] both warpgroups have read step n (frees the dP buffer)
  uint64_t* acc_done = ldd + 2;         // [1]
  uint64_t* mma_drain = acc_done + 1;  // [1] every issued MMA finished (before TMEM is released)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const Geom& g = p.g;
  const int warp = threadIdx.x / 32;
  const int bh = blockIdx.x;
  const int b = bh / g.Hq, h = bh - b * g.Hq;
  const int bkv = b * g.Hkv + h / g.G;
  const int qt = p.n_tiles - 1 - (int)blockIdx.y;  // longest rows first
  const int i0 = qt * BMQ;
  const int ihi = min(i0 + BMQ, g.Lq) - 1;
  // key tiles meeting the band of rows i0 .. ihi (never empty)
  const TileSteps ksteps = row_steps(g, i0, ihi, BN);
  const int nt = ksteps.count();
  constexpr bool two = TWO;  // shared-prefix plan: a row may see two key intervals

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NK; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(k_empty + s, 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(v_full + s, 1);
      mbar_init(v_empty + s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(sdp_full + s, 1);
      mbar_init(ds_full + s, 256);
      mbar_init(ldd + s, 256);  // both warpgroups arrive; the MMA thread only waits
    }
    mbar_init(acc_done, 1);
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (elect_one()) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmG);
      mbar_arrive_expect_tx(q_full, 2 * C::QT_BYTES);
      for (int c = 0; c < KCH; ++c) {
        tma_load_3d(sQ + c * BMQ * 128, &tmQ, q_full, c * 64, i0, bh);
        tma_load_3d(sG + c * BMQ * 128, &tmG, q_full, c * 64, i0, bh);
      }
      // K of each step, the ring refilled as soon as a slot is released
      int nk = 0;
      for (; nk < nt; ++nk) {
        const int j0 = (two ? ksteps.tile(nk) : ksteps.lo0 + nk) * BN;
        const int sk = nk % NK;
        if (nk >= NK && !mbar_wait(k_empty + sk, ((nk / NK) & 1) ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(k_full + sk, C::KV_BYTES);
        for (int c = 0; c < KCH; ++c)
          tma_load_3d(sK + sk * C::KV_BYTES + c * BN * 128, &tmK, k_full + sk, c * 64, j0, bkv);
      }
      if (*abort_flag) {  // unwinding: the loads in flight land before shared memory is released
        mbar_wait_drain(q_full, 0);
        drain_ring(k_full, NK, nk);
      }
    }
  } else if (warp == 10) {
    // V on a warp of its own, so that a wait on one ring never holds up the other
    if (elect_one()) {
      int nv = 0;
      for (; nv < nt; ++nv) {
        const int j0 = (two ? ksteps.tile(nv) : ksteps.lo0 + nv) * BN;
        const int sv = nv % NV;
        if (nv >= NV && !mbar_wait(v_empty + sv, ((nv / NV) & 1) ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(v_full + sv, C::KV_BYTES);
        for (int c = 0; c < KCH; ++c)
          tma_load_3d(sV + sv * C::KV_BYTES + c * BN * 128, &tmV, v_full + sv, c * 64, j0, bkv);
      }
      if (*abort_flag) drain_ring(v_full, NV, nv);
    }
  } else if (warp == 1) {
    if (elect_one()) {
      const uint32_t idS = idesc_f16(BMQ, BN, 0, 0, 0, 0);  // Q x K^T, dO x V^T (both K-major), N = 128
      const uint32_t idQ = idesc_f16(BMQ, D, 0, 0, 0, 1);   // dS (TMEM) x K (MN-major)
      const uint64_t qdk = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t gdk = smem_desc_sw128(smem_u32(sG), 16, 1024);
      bool ok = mbar_wait(q_full, 0, abort_flag);
      auto issue_s = [&](int n) -> bool {  // S(n) into buffer n % 2
        if (!mbar_wait(k_full + n % NK, (n / NK) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint64_t kk = smem_desc_sw128(smem_u32(sK + (n % NK) * C::KV_BYTES), 16, 1024);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks & 3) * 32;
          mma_ss(tmem + C::S_COL + (n & 1) * BN, desc_add(qdk, (ks >> 2) * BMQ * 128 + off),
                 desc_add(kk, (ks >> 2) * BN * 128 + off), idS, ks > 0 ? 1u : 0u);
        }
        return true;
      };
      auto issue_dp = [&](int n) -> bool {  // dP(n) into the dP buffer; completes step n's inputs
        if (!mbar_wait(v_full + n % NV, (n / NV) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint64_t vk = smem_desc_sw128(smem_u32(sV + (n % NV) * C::KV_BYTES), 16, 1024);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks & 3) * 32;
          mma_ss(tmem + C::DP_COL, desc_add(gdk, (ks >> 2) * BMQ * 128 + off),
                 desc_add(vk, (ks >> 2) * BN * 128 + off), idS, ks > 0 ? 1u : 0u);
        }
        mma_commit(v_empty + n % NV);
        mma_commit(sdp_full + (n & 1));  // covers S(n), issued earlier
        return true;
      };
      if (ok) ok = issue_s(0) && issue_dp(0);
      if (ok && nt > 1) ok = issue_s(1);
      for (int n = 0; ok && n < nt; ++n) {
        if (n + 1 < nt) {
          // the dP buffer is free once both warpgroups have read dP(n)
          if (!mbar_wait(ldd + (n & 1), (n >> 1) & 1, abort_flag)) { ok = false; break; }
          if (!issue_dp(n + 1)) { ok = false; break; }
        }
        if (!mbar_wait(ds_full + (n & 1), (n >> 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint64_t kmn = smem_desc_sw128(smem_u32(sK + (n % NK) * C::KV_BYTES), BN * 128, 1024);
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks)
          mma_ts(tmem + C::DQ_COL, tmem + C::S_COL + (n & 1) * BN + ks * 8, desc_add(kmn, ks * 2048), idQ,
                 (n > 0 || ks > 0) ? 1u : 0u);
        mma_commit(k_empty + n % NK);
        if (n + 2 < nt && !issue_s(n + 2)) { ok = false; break; }
      }
      if (ok) mma_commit(acc_done);
      // every MMA issued so far has finished before TMEM is released
      mma_commit(mma_drain);
      mbar_wait_drain(mma_drain, 0);
    }
  } else {
    const int wg = (warp - 2) >> 2;  // warps 2-5 / 6-9; warp % 4 fixes the TMEM lane quarter
    const int r = 32 * (warp & 3) + (threadIdx.x & 31);
    const int i = i0 + r;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const float sl2 = g.scale * kLog2e;
    const float2 rs = (i < g.Lq) ? make_float2(p.stats[(size_t)bh * p.Lpad + i],
                                              p.stats[((size_t)g.B * g.Hq + bh) * p.Lpad + i])
                                : make_float2(0.f, 0.f);
    const int cw0 = wg * CW;
    bool ok = true;
    // loop invariants: this row's band, and the bounds every row of the tile shares
    const int4 vrow = row_vis(g, i, 0);
    const int lo_all = band_key_lo(g, ihi), hi_all = band_key_hi(g, i0);
    for (int n = 0; n < nt; ++n) {
      const int sb = n & 1;
      const int j0 = (two ? ksteps.tile(n) : ksteps.lo0 + n) * BN;
      if (!__all_sync(0xffffffffu, mbar_wait(sdp_full + sb, (n >> 1) & 1, abort_flag))) { ok = false; break; }
      tc_fence_after();
      const bool full = two ? rows_tile_full(g, i0, ihi, j0, j0 + BN - 1) : (j0 >= lo_all && j0 + BN - 1 <= hi_all);
      bool both = false;  // visible key columns of row i
      const int4 vv = two ? vis_in_tile(vshift(vrow, j0), BN, &both) : vshift(vrow, j0);
      const bool two_here = two && __any_sync(0xffffffffu, both);
      uint32_t sv[CW], dv[CW];
#pragma unroll
      for (int c = 0; c < CW / 32; ++c) {
        tmem_ld32(tmem + lane_off + C::S_COL + sb * BN + cw0 + c * 32, *reinterpret_cast<uint32_t(*)[32]>(sv + c * 32));
        tmem_ld32(tmem + lane_off + C::DP_COL + cw0 + c * 32, *reinterpret_cast<uint32_t(*)[32]>(dv + c * 32));
      }
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(ldd + sb);  // also releases the dP buffer to the MMA thread
      // the other warpgroup's packed dS lands on columns this one reads: wait for both
      if (!__all_sync(0xffffffffu, mbar_wait(ldd + sb, (n >> 1) & 1, abort_flag))) { ok = false; break; }
#pragma unroll
      for (int c = 0; c < CW / 32; ++c) {
        const uint32_t(&svc)[32] = *reinterpret_cast<const uint32_t(*)[32]>(sv + c * 32);
        const uint32_t(&dvc)[32] = *reinterpret_cast<const uint32_t(*)[32]>(dv + c * 32);
        const int cb = cw0 + c * 32;
        uint32_t dd[16];
        if (full) dq_chunk<true>(svc, dvc, sl2, rs.x, rs.y, cb, vv, dd);
        else if (two_here) dq_chunk<false, true>(svc, dvc, sl2, rs.x, rs.y, cb, vv, dd);
        else dq_chunk<false>(svc, dvc, sl2, rs.x, rs.y, cb, vv, dd);
        tmem_st16(tmem + lane_off + C::S_COL + sb * BN + cb / 2, dd);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(ds_full + sb);
    }
    if (ok && __all_sync(0xffffffffu, mbar_wait(acc_done, 0, abort_flag))) {
      tc_fence_after();
      // each warpgroup writes half the columns, through TMA stores staged in
      // 16 KB per warp of the (all consumed) dO tile and K / V stages
      const float mul = g.scale * p.stats[dscale_offset(g, p.Lpad) + 1];  // scale / s
      tmem_rows_store_tma(&tmO, tmem + lane_off + C::DQ_COL + wg * (D / 2), wg * (D / 2), D / 2, mul,
                          smem_u32(base) + (uint32_t)(warp - 2) * 16384u, i - (int)(threadIdx.x & 31), bh,
                          (int)(threadIdx.x & 31));
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) atomicCAS(p.status, 0, kStatusTimeout);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t bwd_tc_d(const Geom& g, const uint16_t* q16, const uint16_t* k16, const uint16_t* v16,
                     const uint16_t* g16, const float* stats, int Lpad, float* dq, float* dk, float* dv, int* status,
                     cudaStream_t s, int which) {
  cudaError_t e;
  BwdParams p;
  p.g = g;
  p.stats = stats;
  p.x16 = nullptr;
  p.Lpad = Lpad;
  p.status = status;
  if (which == 0) {
    if constexpr (D <= 128) {
      using C = Kv128Cfg<D>;
      CUtensorMap tq, tk, tv, tg;
      cudaError_t e2;
      if ((e2 = make_tmap_f16(&tq, q16, D, g.Lq, g.B * g.Hq, C::BM)) != cudaSuccess) return e2;
      if ((e2 = make_tmap_f16(&tg, g16, D, g.Lq, g.B * g.Hq, C::BM)) != cudaSuccess) return e2;
      if ((e2 = make_tmap_f16(&tk, k16, D, g.L, g.B * g.Hkv, C::BNK)) != cudaSuccess) return e2;
      if ((e2 = make_tmap_f16(&tv, v16, D, g.L, g.B * g.Hkv, C::BNK)) != cudaSuccess) return e2;
      auto kern = g.Rc > 0 ? dkdv128_tc_kernel<D, true> : dkdv128_tc_kernel<D, false>;
      if ((e2 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM)) !=
          cudaSuccess)
        return e2;
      BwdParams pm = p;
      pm.out0 = dk;
      pm.out1 = dv;
      pm.n_tiles = (g.L + C::BNK - 1) / C::BNK;
      dim3 grid(g.B * g.Hkv, pm.n_tiles);
      CUtensorMap tdk, tdv;
      if ((e2 = make_tmap_f32_out(&tdk, dk, D, g.L, g.B * g.Hkv)) != cudaSuccess) return e2;
      if ((e2 = make_tmap_f32_out(&tdv, dv, D, g.L, g.B * g.Hkv)) != cudaSuccess) return e2;
      kern<<<grid, kThreadsKv128, C::SMEM, s>>>(tq, tk, tv, tg, tdk, tdv, pm);
      return cudaGetLastError();
    } else {
      using C = Kv256PairCfg;
      CUtensorMap tq, tk, tv, tg;
      if ((e = make_tmap_f16(&tq, q16, D, g.Lq, g.B * g.Hq, C::BM)) != cudaSuccess) return e;
      if ((e = make_tmap_f16(&tg, g16, D, g.Lq, g.B * g.Hq, C::BM)) != cudaSuccess) return e;
      if ((e = make_tmap_f16(&tk, k16, D, g.L, g.B * g.Hkv, C::BNK)) != cudaSuccess) return e;
      if ((e = make_tmap_f16(&tv, v16, D, g.L, g.B * g.Hkv, C::BNK)) != cudaSuccess) return e;
      auto kern = g.Rc > 0 ? dkdv256_pair_kernel<true> : dkdv256_pair_kernel<false>;
      if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM)) != cudaSuccess)
        return e;
      BwdParams pm = p;
      pm.out0 = dk;
      pm.out1 = dv;
      pm.n_tiles = (g.L + C::BNK - 1) / C::BNK;
      dim3 grid(2 * g.B * g.Hkv, pm.n_tiles);  // clusters of 2 along x: (dV CTA, dK CTA) of a key tile
      CUtensorMap tdk, tdv;
      if ((e = make_tmap_f32_out(&tdk, dk, D, g.L, g.B * g.Hkv)) != cudaSuccess) return e;
      if ((e = make_tmap_f32_out(&tdv, dv, D, g.L, g.B * g.Hkv)) != cudaSuccess) return e;
      kern<<<grid, kPairThreads, C::SMEM, s>>>(tq, tk, tv, tg, tdk, tdv, pm);
      return cudaGetLastError();
    }
  } else if constexpr (D <= 128) {
    using C = Dq128Cfg<D>;
    CUtensorMap tq, tk, tv, tg;
    if ((e = make_tmap_f16(&tq, q16, D, g.Lq, g.B * g.Hq, C::BMQ)) != cudaSuccess) return e;
    if ((e = make_tmap_f16(&tg, g16, D, g.Lq, g.B * g.Hq, C::BMQ)) != cudaSuccess) return e;
    if ((e = make_tmap_f16(&tk, k16, D, g.L, g.B * g.Hkv, C::BN)) != cudaSuccess) return e;
    if ((e = make_tmap_f16(&tv, v16, D, g.L, g.B * g.Hkv, C::BN)) != cudaSuccess) return e;
    auto kern = g.Rc > 0 ? dq128_tc_kernel<D, true> : dq128_tc_kernel<D, false>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM)) != cudaSuccess)
      return e;
    p.out0 = dq;
    p.out1 = nullptr;
    p.n_tiles = (g.Lq + C::BMQ - 1) / C::BMQ;
    dim3 grid(g.B * g.Hq, p.n_tiles);
    CUtensorMap tdq;
    if ((e = make_tmap_f32_out(&tdq, dq, D, g.Lq, g.B * g.Hq)) != cudaSuccess) return e;
    kern<<<grid, kThreadsKv128, C::SMEM, s>>>(tq, tk, tv, tg, tdq, p);
  } else {
    using C = DqCfg<D>;
    CUtensorMap tk, tv, tg;
    if ((e = make_tmap_f16(&tg, g16, D, g.Lq, g.B * g.Hq, C::BMQ)) != cudaSuccess) return e;
    if ((e = make_tmap_f16_chunks(&tk, k16, D, g.L, g.B * g.Hkv, C::BN, C::KCH)) != cudaSuccess) return e;
    if ((e = make_tmap_f16_chunks(&tv, v16, D, g.L, g.B * g.Hkv, C::BN, C::KCH)) != cudaSuccess) return e;
    auto kern = g.Rc > 0 ? dq_tc_kernel<D, true> : dq_tc_kernel<D, false>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM)) != cudaSuccess)
      return e;
    p.out0 = dq;
    p.out1 = nullptr;
    p.x16 = q16;
    p.n_tiles = (g.Lq + C::BMQ - 1) / C::BMQ;
    dim3 grid(g.B * g.Hq, p.n_tiles);
    CUtensorMap tdq;
    if ((e = make_tmap_f32_out(&tdq, dq, D, g.Lq, g.B * g.Hq)) != cudaSuccess) return e;
    kern<<<grid, kThreads, C::SMEM, s>>>(tk, tv, tg, tdq, p);
  }
  return cudaGetLastError();
}

}  // namespace

bool bwd_tc_supported(int D) { return D == 64 || D == 128 || D == 256 || D == 512; }

int scratch_layout_bwd256() {
  int n0 = 0, n1 = 0, nsm = 0, dev = 0;
  const size_t smem = Kv256PairCfg::SMEM;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev))
    return -1;
  if (cudaFuncSetAttribute(dkdv256_pair_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) ||
      cudaFuncSetAttribute(dkdv256_pair_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n0, dkdv256_pair_kernel<false>, kPairThreads, smem) ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n1, dkdv256_pair_kernel<true>, kPairThreads, smem))
    return -1;
  return (n0 == 1 && n1 == 1 && nsm <= kPairScratchSms) ? 0 : 1;
}

cudaError_t launch_bwd_dscale(const Geom& g, int Lpad, const uint16_t* dO, float* stats, cudaStream_t s) {
  const long long n16 = (long long)g.B * g.Hq * g.Lq * g.D / 8;
  uint32_t* partial = reinterpret_cast<uint32_t*>(stats + dscale_offset(g, Lpad) + 4);
  int* counters = reinterpret_cast<int*>(stats + dscale_offset(g, Lpad) + kWorkCounterFloat);
  bwd_dscale_kernel<<<kAbsmaxBlocks, 256, 0, s>>>(reinterpret_cast<const uint4*>(dO), n16, partial, counters);
  return cudaGetLastError();
}

cudaError_t launch_sink_grad(const Geom& g, int Lpad, const float* stats, float* dsinks, cudaStream_t s) {
  if (!g.sinks) return cudaErrorInvalidValue;
  sink_grad_kernel<<<g.Hq, 256, 0, s>>>(stats, Lpad, g.B, g.Hq, g.Lq, g.sinks, dsinks,
                                        (long long)dscale_offset(g, Lpad));
  return cudaGetLastError();
}

int bwd_stats_lpad(int L) { return (L + 127) / 128 * 128; }

cudaError_t launch_bwd_prep(const Geom& g, int Lpad, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                            const uint16_t* dO, const float* o, const float* lse, uint16_t* q16, uint16_t* k16,
                            uint16_t* v16, uint16_t* g16, float* stats, int* status, cudaStream_t s) {
  PrepParams p;
  p.src[0] = q;
  p.src[1] = k;
  p.src[2] = v;
  p.dst[0] = q16;
  p.dst[1] = k16;
  p.dst[2] = v16;
  p.n[0] = (long long)g.B * g.Hq * g.Lq * g.D;
  p.n[1] = p.n[2] = (long long)g.B * g.Hkv * g.L * g.D;
  p.BH = g.B * g.Hq;
  p.L = g.Lq;
  p.Lpad = Lpad;
  p.D = g.D;
  p.o = o;
  p.dO = dO;
  p.g16 = g16;
  p.lse = lse;
  p.stats = stats;
  p.dscale = stats + dscale_offset(g, Lpad);
  p.status = status;
  // about 8 resident blocks of 256 threads per SM over the four segments
  const long rows = (long)p.BH * Lpad;
  long blocks = (rows + 7) / 8;
  if (blocks > 152L * 4) blocks = 152L * 4;
  if (blocks < 1) blocks = 1;
  bwd_prep_kernel<<<dim3((unsigned)blocks, 4), 256, 0, s>>>(p);
  return cudaGetLastError();
}


cudaError_t launch_bwd_dkdv_tc(const Geom& g, const uint16_t* q16, const uint16_t* k16, const uint16_t* v16,
                               const uint16_t* g16, const float* stats, int Lpad, float* dk, float* dv,
                               int* status, cudaStream_t s) {
  switch (g.D) {
    case 64: return bwd_tc_d<64>(g, q16, k16, v16, g16, stats, Lpad, nullptr, dk, dv, status, s, 0);
    case 128: return bwd_tc_d<128>(g, q16, k16, v16, g16, stats, Lpad, nullptr, dk, dv, status, s, 0);
    case 256: return bwd_tc_d<256>(g, q16, k16, v16, g16, stats, Lpad, nullptr, dk, dv, status, s, 0);
    case 512: return launch_bwd_dkdv_tc512(g, q16, k16, v16, g16, stats, Lpad, dk, dv, status, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bwd_dq_tc(const Geom& g, const uint16_t* q16, const uint16_t* k16, const uint16_t* v16,
                             const uint16_t* g16, const float* stats, int Lpad, float* dq, int* status,
                             cudaStream_t s) {
  switch (g.D) {
    case 64: return bwd_tc_d<64>(g, q16, k16, v16, g16, stats, Lpad, dq, nullptr, nullptr, status, s, 1);
    case 128: return bwd_tc_d<128>(g, q16, k16, v16, g16, stats, Lpad, dq, nullptr, nullptr, status, s, 1);
    case 256: return bwd_tc_d<256>(g, q16, k16, v16, g16, stats, Lpad, dq, nullptr, nullptr, status, s, 1);
    case 512: return launch_bwd_dq_tc512(g, q16, k16, v16, g16, stats, Lpad, dq, status, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace swa
