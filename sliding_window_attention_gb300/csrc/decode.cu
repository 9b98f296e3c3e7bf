// Forward for a few query rows per kv head: a decode step over a KV cache
// (Lq = 1, or a short suffix), with grouped-query heads packed together.
//
// The G query heads of a kv head are consecutive heads, so their Lq query rows
// are M = G * Lq consecutive rows of q ([B * Hkv, M, D] viewed that way); one
// CTA takes all M rows and a chunk of the keys in band, so every K and V row
// is read from HBM once per kv head ("MiniCPM5 Decode Megakernel -- end-to-end
// build plan", section 4.1 stage 5: query head h reads kv head h / (Hq/Hkv)).
// Query row i sits at key position i + Lk - Lq and sees the keys of its band
// ("Lab 028 lab detail: Off NVIDIA, you fix the platform yourself", "Plan for
// the build" step 4 and "What I changed, in plain terms" items 3-4).
//
// With M <= 16 rows the work is a stream over the cache with about 2 M flops
// per byte, far below the tensor-core ridge, so it runs on the CUDA cores in
// fp32 on the bf16 inputs: TMA brings 32 KB K and V blocks (128-byte swizzle,
// double-buffered) into shared memory; per block the scores are partial dot
// products over 64-column segments (a warp = 32 keys x one segment, so each
// lane reads its own key row and the query values are warp-wide broadcasts),
// an online softmax per row (one warp per row), then O += P V (a thread per
// head-dim column).  The key range is split into chunks over about two waves
// of CTAs; a second kernel merges the chunks' (max, sum, unnormalised O).
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "swa_internal.h"
#include "tc_ptx.cuh"

namespace swa {
namespace {

using namespace tc;

constexpr int kThr = 256;
constexpr int kMaxRows = kDecodeMaxRows;  // M = G * Lq
constexpr int kBlockElems = 32 * 512;     // keys per block x D: one 32 KB bf16 K (or V) block
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct DecParams {
  Geom g;
  const uint16_t* q;  // bf16, [B * Hkv, M, D]
  float* o;           // fp32, [B * Hkv, M, D]
  float* lse;         // fp32, [B * Hkv, M]
  float* part_o;      // [n_chunks][B * Hkv][M][D] unnormalised O of each chunk
  float* part_ml;     // [n_chunks][B * Hkv][M][2]: running max (log2 units), sum
  int M;
  int k_begin, k_end;  // keys any row of the group sees: [k_begin, k_end)
  int chunk;           // keys per chunk (a multiple of the block)
  int n_chunks;
  int* status;
};

template <int D>
struct DecCfg {
  static constexpr int NSEG = D / 64;             // 64-column segments of a row
  static constexpr int KB = kBlockElems / D;      // keys per block: 32 (D = 512) .. 256 (D = 64)
  static constexpr int BLK = KB * D * 2;          // 32 KB
  static constexpr int OFF_Q = 4 * BLK;           // K, V double buffers first
  static constexpr int OFF_PART = OFF_Q + kMaxRows * D * 4;
  static constexpr int OFF_P = OFF_PART + NSEG * kMaxRows * KB * 4;
  static constexpr int OFF_ALPHA = OFF_P + kMaxRows * KB * 4;
  static constexpr int OFF_BAR = OFF_ALPHA + kMaxRows * 4;
  static constexpr size_t SMEM = (size_t)OFF_BAR + 64 + 1024;
  // the end-of-chunk reduction over key subsets reuses the scratch from OFF_PART
  static constexpr int KSUB = D >= 256 ? 1 : 256 / D;  // key subsets in the O += P V phase
  static constexpr int DPT = D >= 256 ? D / 256 : 1;   // head-dim columns per thread
  static_assert(OFF_ALPHA - OFF_PART >= KSUB * kMaxRows * D * 4 || KSUB == 1, "subset reduction scratch");
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(8 % NSEG == 0 && KB % 32 == 0, "warp tiling of the score phase");
};

// bf16 pair (one 32-bit word) to two floats
__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

template <int D>
__global__ void __launch_bounds__(kThr, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const DecParams p) {
  using C = DecCfg<D>;
  constexpr int NSEG = C::NSEG, KB = C::KB, KSUB = C::KSUB, DPT = C::DPT;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* qs = reinterpret_cast<float*>(base + C::OFF_Q);        // [M][D] scale * log2(e) * q
  float* part = reinterpret_cast<float*>(base + C::OFF_PART);   // [NSEG][kMaxRows][KB] partial scores
  float* ps = reinterpret_cast<float*>(base + C::OFF_P);        // [kMaxRows][KB] P of the block
  float* alph = reinterpret_cast<float*>(base + C::OFF_ALPHA);  // [kMaxRows] rescale of O for the block
  uint64_t* full = reinterpret_cast<uint64_t*>(base + C::OFF_BAR);  // [2]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + 2);

  const Geom& g = p.g;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
  const int M = p.M;
  const int bkv = blockIdx.y;  // b * Hkv + kv head
  const int c0 = p.k_begin + (int)blockIdx.x * p.chunk;
  const int c1 = min(p.k_end, c0 + p.chunk);
  const int nb = (c1 - c0 + KB - 1) / KB;  // blocks of this chunk (>= 1)

  if (tid == 0) {
    mbar_init(full + 0, 1);
    mbar_init(full + 1, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // the group's query rows, pre-scaled so that scores come out in log2 units
  const float sl2 = g.scale * kLog2e;
  const uint16_t* qg = p.q + (size_t)bkv * M * D;
  for (int e = tid; e < M * D; e += kThr) qs[e] = __uint_as_float((uint32_t)qg[e] << 16) * sl2;
  __syncthreads();
  auto issue = [&](int blk) {
    const int buf = blk & 1;
    mbar_arrive_expect_tx(full + buf, 2 * C::BLK);
    tma_load_4d(base + buf * C::BLK, &tmK, full + buf, 0, c0 + blk * KB, 0, bkv);
    tma_load_4d(base + (2 + buf) * C::BLK, &tmV, full + buf, 0, c0 + blk * KB, 0, bkv);
  };
  if (tid == 0) {
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    issue(0);
  }

  // per-row softmax state, held by the warp that owns the row (rows w, w + 8)
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  // O accumulators: thread t owns head-dim columns [DPT * (t % (D / DPT)), +DPT) for key subset t / (D / DPT)
  constexpr int DCOLS = D / DPT;  // threads per key subset
  const int dcol = (tid % DCOLS) * DPT, ksub = tid / DCOLS;
  float acc[kMaxRows][DPT];
#pragma unroll
  for (int m = 0; m < kMaxRows; ++m)
#pragma unroll
    for (int e = 0; e < DPT; ++e) acc[m][e] = 0.f;

  int issued = 1;
  bool ok = true;
  for (int blk = 0; blk < nb; ++blk) {
    const int buf = blk & 1;
    if (tid == 0 && blk + 1 < nb) {
      issue(blk + 1);  // buffer buf ^ 1 held block blk - 1, fully consumed before the last barrier
      ++issued;
    }
    if (!__syncthreads_and(mbar_wait(full + buf, (blk >> 1) & 1, abort_flag))) { ok = false; break; }
    const unsigned char* kb = base + buf * C::BLK;
    const unsigned char* vb = base + (2 + buf) * C::BLK;
    const int kbase = c0 + blk * KB;  // key index of the block's row 0

    // ---- scores: warp w = (key group w / NSEG, segment w % NSEG), lane = key of the group
    for (int kg = warp / NSEG; kg < KB / 32; kg += 8 / NSEG) {
      const int seg = warp % NSEG, kl = kg * 32 + lane;
      // the key row's 64 columns of this segment: eight 16-byte chunks, 128-byte swizzle
      const unsigned char* row = kb + seg * (KB * 128) + kl * 128;
      float kv[64];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 w = *reinterpret_cast<const uint4*>(row + ((c ^ (kl & 7)) << 4));
        const float2 a = bf2_to_f2(w.x), b = bf2_to_f2(w.y), cc = bf2_to_f2(w.z), d = bf2_to_f2(w.w);
        kv[8 * c + 0] = a.x;
        kv[8 * c + 1] = a.y;
        kv[8 * c + 2] = b.x;
        kv[8 * c + 3] = b.y;
        kv[8 * c + 4] = cc.x;
        kv[8 * c + 5] = cc.y;
        kv[8 * c + 6] = d.x;
        kv[8 * c + 7] = d.y;
      }
      for (int m = 0; m < M; ++m) {
        const float4* qr = reinterpret_cast<const float4*>(qs + m * D + seg * 64);
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const float4 qa = qr[e], qb = qr[e + 1];  // the same address in every lane: a broadcast
          s0 = fmaf(qa.x, kv[4 * e + 0], s0);
          s0 = fmaf(qa.y, kv[4 * e + 1], s0);
          s0 = fmaf(qa.z, kv[4 * e + 2], s0);
          s0 = fmaf(qa.w, kv[4 * e + 3], s0);
          s1 = fmaf(qb.x, kv[4 * e + 4], s1);
          s1 = fmaf(qb.y, kv[4 * e + 5], s1);
          s1 = fmaf(qb.z, kv[4 * e + 6], s1);
          s1 = fmaf(qb.w, kv[4 * e + 7], s1);
        }
        part[(seg * kMaxRows + m) * KB + kl] = s0 + s1;
      }
    }
    __syncthreads();

    // ---- online softmax: warp w owns rows w and w + 8
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int m = warp + 8 * rr;
      if (m >= M) break;
      const int i = m % g.Lq;  // query row of this packed row
      const int lo = max(band_key_lo(g, i), c0), hi = min(band_key_hi(g, i), c1 - 1);
      float sv[KB / 32];
      float mx = -INFINITY;
#pragma unroll
      for (int t = 0; t < KB / 32; ++t) {
        const int kl = lane + 32 * t, key = kbase + kl;
        float s = 0.f;
#pragma unroll
        for (int seg = 0; seg < NSEG; ++seg) s += part[(seg * kMaxRows + m) * KB + kl];
        s = (key >= lo && key <= hi) ? s : -INFINITY;
        sv[t] = s;
        mx = fmaxf(mx, s);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_new = fmaxf(m_run[rr], mx);
      // no key seen yet: nothing to rescale, and P = 0
      const float alpha = (m_run[rr] == -INFINITY) ? 1.f : exp2f(m_run[rr] - m_new);
      float sum = 0.f;
#pragma unroll
      for (int t = 0; t < KB / 32; ++t) {
        const float pv = (sv[t] == -INFINITY) ? 0.f : exp2f(sv[t] - m_new);
        ps[m * KB + lane + 32 * t] = pv;
        sum += pv;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      l_run[rr] = l_run[rr] * alpha + sum;
      m_run[rr] = m_new;
      if (lane == 0) alph[m] = alpha;
    }
    __syncthreads();

    // ---- O += P V: thread = (key subset, head-dim columns)
    {
      const int seg = dcol / 64, cb = (dcol % 64) * 2;  // byte offset of the columns in a 128-byte row
#pragma unroll
      for (int m = 0; m < kMaxRows; ++m) {
        if (m < M) {
          const float a = alph[m];
#pragma unroll
          for (int e = 0; e < DPT; ++e) acc[m][e] *= a;
        }
      }
      for (int kl = ksub; kl < KB; kl += KSUB) {
        const unsigned char* row = vb + seg * (KB * 128) + kl * 128;
        const unsigned char* src = row + ((((cb >> 4) ^ (kl & 7)) << 4) | (cb & 15));
        float vv[DPT];
        if constexpr (DPT == 2) {
          const float2 f = bf2_to_f2(*reinterpret_cast<const uint32_t*>(src));
          vv[0] = f.x;
          vv[1] = f.y;
        } else {
          vv[0] = __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t*>(src)) << 16);
        }
#pragma unroll
        for (int m = 0; m < kMaxRows; ++m) {
          if (m < M) {
            const float pv = ps[m * KB + kl];  // the same address in every lane: a broadcast
#pragma unroll
            for (int e = 0; e < DPT; ++e) acc[m][e] = fmaf(pv, vv[e], acc[m][e]);
          }
        }
      }
    }
    __syncthreads();  // part, ps, alph and this block's buffer are free again
  }
  ok = __syncthreads_and(ok && !*abort_flag);

  if (ok) {
    // sum the key subsets' accumulators (head dims below 256), through the score scratch
    if constexpr (KSUB > 1) {
      float* red = part;  // [KSUB][kMaxRows][D]
#pragma unroll
      for (int m = 0; m < kMaxRows; ++m)
        if (m < M) red[(ksub * kMaxRows + m) * D + dcol] = acc[m][0];
      __syncthreads();
      if (ksub == 0) {
#pragma unroll
        for (int m = 0; m < kMaxRows; ++m) {
          if (m < M) {
            float t = 0.f;
            for (int s = 0; s < KSUB; ++s) t += red[(s * kMaxRows + m) * D + dcol];
            acc[m][0] = t;
          }
        }
      }
    }
    // row statistics to shared memory (the owning warps hold them)
    float* mls = ps;  // [kMaxRows][2], the P scratch is free
    if (lane == 0) {
      if (warp < M) {
        mls[2 * warp] = m_run[0];
        mls[2 * warp + 1] = l_run[0];
      }
      if (warp + 8 < M) {
        mls[2 * (warp + 8)] = m_run[1];
        mls[2 * (warp + 8) + 1] = l_run[1];
      }
    }
    __syncthreads();
    if (ksub == 0) {
      if (p.n_chunks == 1) {
        // the only chunk: normalise and write the result
#pragma unroll
        for (int m = 0; m < kMaxRows; ++m) {
          if (m < M) {
            const float inv = 1.f / mls[2 * m + 1];
            float* orow = p.o + ((size_t)bkv * M + m) * D + dcol;
#pragma unroll
            for (int e = 0; e < DPT; ++e) orow[e] = acc[m][e] * inv;
          }
        }
        if (tid < M) p.lse[(size_t)bkv * M + tid] = (mls[2 * tid] + log2f(mls[2 * tid + 1])) * kLn2;
      } else {
        const size_t cb = (size_t)blockIdx.x * gridDim.y + bkv;
#pragma unroll
        for (int m = 0; m < kMaxRows; ++m) {
          if (m < M) {
            float* orow = p.part_o + (cb * M + m) * D + dcol;
#pragma unroll
            for (int e = 0; e < DPT; ++e) orow[e] = acc[m][e];
          }
        }
        if (tid < M) {
          p.part_ml[(cb * M + tid) * 2] = mls[2 * tid];
          p.part_ml[(cb * M + tid) * 2 + 1] = mls[2 * tid + 1];
        }
      }
    }
  }
  // unwinding: the loads in flight land before shared memory is released
  if (*abort_flag && tid == 0) {
    for (int k = issued - 1; k >= 0 && k >= issued - 2; --k) mbar_wait_drain(full + (k & 1), (k >> 1) & 1);
    atomicCAS(p.status, 0, kStatusTimeout);
  }
  __syncthreads();
}

// Merge of the chunks of one packed row (b * Hkv + kv head, m): with
// w_c = 2^(max_c - max), o = sum_c w_c O_c / sum_c w_c l_c and
// lse = (max + log2 sum_c w_c l_c) ln 2.  One block per row, a thread per
// head-dim column.
__global__ void __launch_bounds__(128) decode_combine_kernel(DecParams p, int D) {
  const int row = blockIdx.x;  // (b * Hkv + kv head) * M + m
  const int rows = gridDim.x;
  float mx = -INFINITY;
  for (int c = 0; c < p.n_chunks; ++c) mx = fmaxf(mx, p.part_ml[((size_t)c * rows + row) * 2]);
  float l = 0.f;
  for (int c = 0; c < p.n_chunks; ++c) {
    const float mc = p.part_ml[((size_t)c * rows + row) * 2];
    if (mc != -INFINITY) l += exp2f(mc - mx) * p.part_ml[((size_t)c * rows + row) * 2 + 1];
  }
  const float inv = 1.f / l;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float t = 0.f;
    for (int c = 0; c < p.n_chunks; ++c) {
      const float mc = p.part_ml[((size_t)c * rows + row) * 2];
      if (mc != -INFINITY) t = fmaf(exp2f(mc - mx), p.part_o[((size_t)c * rows + row) * D + d], t);
    }
    p.o[(size_t)row * D + d] = t * inv;
  }
  if (threadIdx.x == 0) p.lse[row] = (mx + log2f(l)) * kLn2;
}

// Key range of the group and its split into chunks of whole blocks, aiming at
// about two waves of CTAs on 152 SMs.
struct DecPlan {
  int k_begin, k_end, chunk, n_chunks;
};
DecPlan decode_plan(const Geom& g) {
  DecPlan pl;
  pl.k_begin = band_key_lo(g, 0);
  pl.k_end = band_key_hi(g, g.Lq - 1) + 1;
  const int KB = kBlockElems / g.D;
  const int range = pl.k_end - pl.k_begin;
  const int groups = g.B * g.Hkv;
  int want = (2 * 152 + groups - 1) / groups;
  const int max_chunks = (range + KB - 1) / KB;
  if (want > max_chunks) want = max_chunks;
  if (want < 1) want = 1;
  pl.chunk = ((range + want - 1) / want + KB - 1) / KB * KB;
  pl.n_chunks = (range + pl.chunk - 1) / pl.chunk;
  return pl;
}

template <int D>
cudaError_t decode_d(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v, float* o, float* lse,
                     float* ws, int* status, cudaStream_t s) {
  using C = DecCfg<D>;
  CUtensorMap tk, tv;
  cudaError_t e;
  // one TMA instruction per 32 KB block: all D / 64 segments of KB key rows
  if ((e = make_tmap_f16_chunks(&tk, k, D, g.L, g.B * g.Hkv, C::KB, C::NSEG)) != cudaSuccess) return e;
  if ((e = make_tmap_f16_chunks(&tv, v, D, g.L, g.B * g.Hkv, C::KB, C::NSEG)) != cudaSuccess) return e;
  const DecPlan pl = decode_plan(g);
  DecParams p;
  p.g = g;
  p.q = q;
  p.o = o;
  p.lse = lse;
  p.M = g.G * g.Lq;
  p.k_begin = pl.k_begin;
  p.k_end = pl.k_end;
  p.chunk = pl.chunk;
  p.n_chunks = pl.n_chunks;
  p.part_o = ws;
  p.part_ml = ws + (size_t)pl.n_chunks * g.B * g.Hkv * p.M * D;
  p.status = status;
  auto kern = decode_kernel<D>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM)) != cudaSuccess)
    return e;
  kern<<<dim3(pl.n_chunks, g.B * g.Hkv), kThr, C::SMEM, s>>>(tk, tv, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (pl.n_chunks > 1) {
    decode_combine_kernel<<<g.B * g.Hkv * p.M, 128, 0, s>>>(p, D);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace

bool decode_supported(const Geom& g) { return g.G * g.Lq <= kDecodeMaxRows; }

size_t decode_workspace_bytes(const Geom& g) {
  const DecPlan pl = decode_plan(g);
  if (pl.n_chunks <= 1) return 0;
  const size_t rows = (size_t)pl.n_chunks * g.B * g.Hkv * g.G * g.Lq;
  return rows * ((size_t)g.D + 2) * sizeof(float);
}

cudaError_t launch_fwd_decode(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v, float* o,
                              float* lse, float* ws, int* status, cudaStream_t s) {
  switch (g.D) {
    case 64: return decode_d<64>(g, q, k, v, o, lse, ws, status, s);
    case 128: return decode_d<128>(g, q, k, v, o, lse, ws, status, s);
    case 256: return decode_d<256>(g, q, k, v, o, lse, ws, status, s);
    case 512: return decode_d<512>(g, q, k, v, o, lse, ws, status, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace swa
