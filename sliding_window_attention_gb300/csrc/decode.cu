// Forward for a few query rows per kv head: a decode step over a KV cache
// (Lq = 1, or a short suffix), with grouped-query heads packed together.
//
// The G query heads of a kv head are consecutive heads, so their Lq query rows
// are M = G * Lq consecutive rows of q ([B * Hkv, M, D] viewed that way); one
// CTA takes all M <= 16 rows and a chunk of the keys in band, so every K and V
// row is read from HBM once per kv head ("MiniCPM5 Decode Megakernel -- end-to-
// end build plan", section 4.1 stage 5: query head h reads kv head h /
// (Hq/Hkv)).  Query row i sits at key position i + Lk - Lq and sees the keys of
// its band ("Lab 028 lab detail: Off NVIDIA, you fix the platform yourself",
// "Plan for the build" step 4 and "What I changed, in plain terms" items 3-4).
//
// The products are taken transposed, so that the 128 keys of a tile (not the
// few query rows) fill the MMA's M dimension:
//   S^T (128 keys x 16 rows) = K_tile (128 x D) . Q^T        tcgen05, N = 16
//   O^T (D x 16 rows)       += V_tile^T (D x 128) . P^T      tcgen05, per 128 columns of D
// K, V and q are read as bf16 straight from the caller's tensors (no fp16
// copies), so P is rounded to bf16 for the second product (both operands of
// one MMA have one type).  The elementwise warps hold one key (one TMEM lane)
// each: per tile they take the column maxima and sums over the 128 keys
// (shuffles, then a 4-warp exchange), keep the running maximum per row
// lazily (O^T is rescaled only when a maximum grows by more than 2^8), and
// write P^T as the K-major B operand.  K and V arrive in 32 KB slots (two
// 64-column chunks of 128 key rows, one TMA instruction each) through one
// ring, in the order the MMAs consume them.  The key range is split into
// chunks so that all CTAs run in one wave; a second kernel merges the
// chunks' (max, sum, unnormalised O).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "swa_internal.h"
#include "tc_ptx.cuh"

namespace swa {
namespace {

using namespace tc;

constexpr int kThr = 192;   // warp 0 TMA, warp 1 MMA, warps 2-5 elementwise (thread = key = TMEM lane)
constexpr int T = 128;      // keys per tile
constexpr int kNR = kDecodeMaxRows;  // MMA N: the M = G * Lq query rows, padded to 16
constexpr int kSlot = 32 * 1024;  // ring slot: two 64-column chunks of 128 key rows
constexpr int kNSlot = 6;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;

struct DecParams {
  Geom g;
  float* o;           // fp32, [B * Hkv, M, D]
  float* lse;         // fp32, [B * Hkv, M]
  float* part_o;      // [n_chunks][B * Hkv][M][D] unnormalised O of each chunk
  float* part_ml;     // [n_chunks][B * Hkv][M][2]: running max (log2 units), sum
  int M;
  int k_begin, k_end;  // keys any row of the group sees: [k_begin, k_end)
  int chunk;           // keys per chunk (a multiple of the tile)
  int n_chunks;
  int* status;
};

template <int D>
struct DecCfg {
  static constexpr int NCH = D / 64;                  // 64-column chunks of a row
  static constexpr int CPS = NCH < 2 ? NCH : 2;       // chunks per slot
  static constexpr int SPT = NCH / CPS;               // slots per tile and tensor
  static constexpr int NDC = (D + 127) / 128;         // 128-column blocks of O^T
  static constexpr int OFF_Q = kNSlot * kSlot;        // Q: NCH chunks of [16 rows x 128 B]
  static constexpr int OFF_P = OFF_Q + NCH * kNR * 128;  // P^T: 2 buffers of 2 chunks [16 rows x 128 B]
  static constexpr int OFF_RED = OFF_P + 2 * 2 * kNR * 128;  // [2 tile parities][4 warps][16] maxima, then sums
  static constexpr int OFF_BAR = OFF_RED + 2 * 4 * kNR * 4;
  static constexpr size_t SMEM = (size_t)OFF_BAR + 256 + 1024;
  static constexpr uint32_t S_COL = 0, O_COL = 2 * kNR;  // TMEM: S^T buffers [0, 32), O^T blocks from 32
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(O_COL + NDC * kNR <= 128, "TMEM columns");
};

__device__ __forceinline__ uint16_t bf16_bits(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }

template <int D>
__global__ void __launch_bounds__(kThr, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const DecParams p) {
  using C = DecCfg<D>;
  constexpr int NCH = C::NCH, CPS = C::CPS, SPT = C::SPT, NDC = C::NDC;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sQ = base + C::OFF_Q;
  unsigned char* sP = base + C::OFF_P;
  float* red = reinterpret_cast<float*>(base + C::OFF_RED);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::OFF_BAR);
  uint64_t* slot_full = bars;              // [kNSlot]
  uint64_t* slot_empty = slot_full + kNSlot;  // [kNSlot]
  uint64_t* q_full = slot_empty + kNSlot;  // [1]
  uint64_t* s_full = q_full + 1;           // [2] S^T(n) in TMEM
  uint64_t* p_full = s_full + 2;           // [2] P^T(n) written (and O^T rescaled) by the elementwise warps
  uint64_t* o_done = p_full + 2;           // [1] PV(n) finished
  uint64_t* red_bar = o_done + 1;          // [2] the four elementwise warps posted their column maxima (by tile parity)
  uint64_t* fin_bar = red_bar + 2;         // [1] ... their partial row sums
  uint64_t* mma_drain = fin_bar + 1;       // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const Geom& g = p.g;
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int M = p.M;
  const int bkv = blockIdx.y;  // b * Hkv + kv head
  const int c0 = p.k_begin + (int)blockIdx.x * p.chunk;
  const int c1 = min(p.k_end, c0 + p.chunk);
  const int nt = (c1 - c0 + T - 1) / T;  // key tiles of this chunk (>= 1)

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNSlot; ++s) {
      mbar_init(slot_full + s, 1);
      mbar_init(slot_empty + s, 1);
    }
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(s_full + s, 1);
      mbar_init(p_full + s, 128);
    }
    mbar_init(o_done, 1);
    mbar_init(red_bar + 0, 128);
    mbar_init(red_bar + 1, 128);
    mbar_init(fin_bar, 128);
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one()) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      mbar_arrive_expect_tx(q_full, NCH * kNR * 128);
      for (int c = 0; c < NCH; ++c) tma_load_3d(sQ + c * kNR * 128, &tmQ, q_full, c * 64, 0, bkv);
      // slots in MMA order: K(0), K(1), then per tile n: V(n), K(n + 2)
      int issued = 0;
      bool ok = true;
      auto load_tile = [&](const CUtensorMap* m, int n) -> bool {
        for (int sp = 0; sp < SPT; ++sp, ++issued) {
          const int s = issued % kNSlot;
          if (issued >= kNSlot && !mbar_wait(slot_empty + s, ((issued / kNSlot) & 1) ^ 1, abort_flag)) return false;
          mbar_arrive_expect_tx(slot_full + s, CPS * T * 128);
          tma_load_4d(base + s * kSlot, m, slot_full + s, 0, c0 + n * T, sp * CPS, bkv);
        }
        return true;
      };
      ok = load_tile(&tmK, 0) && (nt < 2 || load_tile(&tmK, 1));
      for (int n = 0; ok && n < nt; ++n) ok = load_tile(&tmV, n) && (n + 2 >= nt || load_tile(&tmK, n + 2));
      if (*abort_flag) {  // unwinding: the loads in flight land before shared memory is released
        mbar_wait_drain(q_full, 0);
        drain_ring(slot_full, kNSlot, issued);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      const uint32_t idS = idesc_f16(T, kNR, 1, 1, 0, 0);   // K (K-major) x Q^T (K-major), bf16
      const uint32_t idPV = idesc_f16(T, kNR, 1, 1, 1, 0);  // V^T (MN-major) x P^T (K-major), bf16
      const uint64_t qd = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      int used = 0;
      bool ok = mbar_wait(q_full, 0, abort_flag);
      auto issue_s = [&](int n) -> bool {  // S^T(n) into buffer n & 1
        const uint32_t col = C::S_COL + kNR * (n & 1);
        for (int sp = 0; sp < SPT; ++sp, ++used) {
          const int s = used % kNSlot;
          if (!mbar_wait(slot_full + s, (used / kNSlot) & 1, abort_flag)) return false;
          tc_fence_after();
          const uint64_t kd = smem_desc_sw128(smem_u32(base + s * kSlot), 16, 1024);
#pragma unroll
          for (int cc = 0; cc < CPS; ++cc) {
            const int c = sp * CPS + cc;  // chunk of D
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_ss(tmem + col, desc_add(kd, cc * T * 128 + ks * 32), desc_add(qd, c * kNR * 128 + ks * 32), idS,
                     (c | ks) ? 1u : 0u);
          }
          mma_commit(slot_empty + s);
        }
        mma_commit(s_full + (n & 1));
        return true;
      };
      if (ok) ok = issue_s(0) && (nt < 2 || issue_s(1));
      for (int n = 0; ok && n < nt; ++n) {
        if (!mbar_wait(p_full + (n & 1), (n >> 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint64_t pd = smem_desc_sw128(smem_u32(sP + (n & 1) * 2 * kNR * 128), 16, 1024);
        // O^T block h (head-dim columns [128 h, 128 h + 128)) += V^T . P^T: one slot per block
        for (int h = 0; h < SPT; ++h, ++used) {
          const int s = used % kNSlot;
          if (!mbar_wait(slot_full + s, (used / kNSlot) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint64_t vd = smem_desc_sw128(smem_u32(base + s * kSlot), T * 128, 1024);  // MN-major
#pragma unroll
          for (int ks = 0; ks < T / 16; ++ks)
            mma_ss(tmem + C::O_COL + kNR * h, desc_add(vd, ks * 2048),
                   desc_add(pd, (ks >> 2) * kNR * 128 + (ks & 3) * 32), idPV, (n > 0 || ks > 0) ? 1u : 0u);
          mma_commit(slot_empty + s);
        }
        if (!ok) break;
        mma_commit(o_done);
        if (n + 2 < nt && !issue_s(n + 2)) { ok = false; break; }  // after PV(n): S buffer n & 1 is free
      }
      mma_commit(mma_drain);
      mbar_wait_drain(mma_drain, 0);
    }
  } else {
    // ------------------------------------------------------------ elementwise
    const int q4 = warp & 3;  // TMEM lane quarter of this warp
    const int t = 32 * q4 + lane;  // key of the tile (S^T lane), head-dim row of O^T
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const float sl2 = g.scale * kLog2e;
    // key range of each packed row: row q is query position q % Lq
    int lo[kNR], hi[kNR];
#pragma unroll
    for (int q = 0; q < kNR; ++q) {
      const int i = q < M ? q % g.Lq : 0;
      lo[q] = q < M ? max(band_key_lo(g, i), c0) : 1;
      hi[q] = q < M ? min(band_key_hi(g, i), c1 - 1) : 0;  // padding rows see nothing
    }
    float m_run[kNR], l_part[kNR];
#pragma unroll
    for (int q = 0; q < kNR; ++q) {
      m_run[q] = -INFINITY;
      l_part[q] = 0.f;
    }
    bool ok = true;
    for (int n = 0; n < nt; ++n) {
      const int key = c0 + n * T + t;
      if (!__all_sync(0xffffffffu, mbar_wait(s_full + (n & 1), (n >> 1) & 1, abort_flag))) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[kNR];
      tmem_ld16(tmem + lane_off + C::S_COL + kNR * (n & 1), sr);
      tmem_wait_ld();
      float sv[kNR], mx[kNR];
#pragma unroll
      for (int q = 0; q < kNR; ++q) {
        sv[q] = (key >= lo[q] && key <= hi[q]) ? __uint_as_float(sr[q]) * sl2 : -INFINITY;
        mx[q] = sv[q];
      }
      // column maxima over the 128 keys: the warp, then the four warps
#pragma unroll
      for (int q = 0; q < kNR; ++q)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx[q] = fmaxf(mx[q], __shfl_xor_sync(0xffffffffu, mx[q], o));
      // exchange through shared memory, buffer by tile parity: a warp cannot
      // reach tile n + 2 before every warp has finished tile n (S(n + 2) is
      // issued only after all 128 threads released P(n))
      float* rb = red + (n & 1) * 4 * kNR;
      if (lane < kNR) {
        float v = mx[0];
#pragma unroll
        for (int q = 1; q < kNR; ++q) v = (lane == q) ? mx[q] : v;
        rb[q4 * kNR + lane] = v;
      }
      mbar_arrive(red_bar + (n & 1));  // release: the writes above are visible to the waiters
      if (!__all_sync(0xffffffffu, mbar_wait(red_bar + (n & 1), (n >> 1) & 1, abort_flag))) { ok = false; break; }
      bool grow = false;
      float alpha[kNR];
#pragma unroll
      for (int q = 0; q < kNR; ++q) {
        const float tm = fmaxf(fmaxf(rb[q], rb[kNR + q]), fmaxf(rb[2 * kNR + q], rb[3 * kNR + q]));
        alpha[q] = 1.f;
        if (tm > m_run[q] + kRescaleLog2) {  // the running maximum moves (lazily)
          if (m_run[q] != -INFINITY) {
            alpha[q] = exp2f(m_run[q] - tm);
            grow = true;
          }
          m_run[q] = tm;
        }
      }
      // PV(n - 1) has finished: O^T may be rescaled and P buffer n & 1 (last read by PV(n - 2)) rewritten
      if (n > 0 && !__all_sync(0xffffffffu, mbar_wait(o_done, (n - 1) & 1, abort_flag))) { ok = false; break; }
      tc_fence_after();
      if (grow && n > 0) {  // uniform: every thread holds the same row maxima
#pragma unroll
        for (int h = 0; h < NDC; ++h) {
          uint32_t ov[kNR];
          tmem_ld16(tmem + lane_off + C::O_COL + kNR * h, ov);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < kNR; ++q) ov[q] = __float_as_uint(__uint_as_float(ov[q]) * alpha[q]);
          tmem_st16(tmem + lane_off + C::O_COL + kNR * h, ov);
        }
        tmem_wait_st();
      }
      // P^T(n) as the K-major B operand: row q, key t -> chunk t / 64, 128-byte swizzle
      unsigned char* pb = sP + (n & 1) * 2 * kNR * 128 + (t >> 6) * kNR * 128;
      const int kc = t & 63;
#pragma unroll
      for (int q = 0; q < kNR; ++q) {
        const float pv = (sv[q] == -INFINITY || m_run[q] == -INFINITY) ? 0.f : exp2f(sv[q] - m_run[q]);
        l_part[q] = l_part[q] * alpha[q] + pv;
        const int off = q * 128 + ((((kc >> 3) ^ (q & 7))) << 4) + (kc & 7) * 2;
        *reinterpret_cast<uint16_t*>(pb + off) = bf16_bits(pv);
      }
      fence_proxy_async_smem();  // generic writes -> the tensor core's reads
      tc_fence_before();
      mbar_arrive(p_full + (n & 1));
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(o_done, (nt - 1) & 1, abort_flag));
    if (ok) {
      // row sums: the partial sums of the 128 threads, exchanged through the
      // buffer of parity nt & 1 (its last readers finished tile nt - 2 or
      // earlier, before any thread got here)
#pragma unroll
      for (int q = 0; q < kNR; ++q)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l_part[q] += __shfl_xor_sync(0xffffffffu, l_part[q], o);
      float* rb = red + (nt & 1) * 4 * kNR;
      if (lane < kNR) {
        float v = l_part[0];
#pragma unroll
        for (int q = 1; q < kNR; ++q) v = (lane == q) ? l_part[q] : v;
        rb[q4 * kNR + lane] = v;
      }
      mbar_arrive(fin_bar);
      ok = __all_sync(0xffffffffu, mbar_wait(fin_bar, 0, abort_flag));
    }
    ok = __all_sync(0xffffffffu, ok && !*abort_flag);
    if (ok) {
      tc_fence_after();
      const float* rb = red + (nt & 1) * 4 * kNR;
      float l_tot[kNR];
#pragma unroll
      for (int q = 0; q < kNR; ++q) l_tot[q] = (rb[q] + rb[kNR + q]) + (rb[2 * kNR + q] + rb[3 * kNR + q]);
      const bool single = p.n_chunks == 1;
      const size_t cb = (size_t)blockIdx.x * gridDim.y + bkv;
      // a single chunk finishes the rows here: 1 / l, or with attention
      // sinks the factor that folds the row's head sink into the normaliser
      float fac[kNR], lse_row[kNR];
#pragma unroll
      for (int q = 0; q < kNR; ++q) {
        fac[q] = 1.f / l_tot[q];
        lse_row[q] = (m_run[q] + log2f(l_tot[q])) * kLn2;
        if (single && g.sinks && q < M)
          fac[q] = sink_finish(g.sinks[(bkv % g.Hkv) * g.G + q / g.Lq], m_run[q], l_tot[q], &lse_row[q]);
      }
#pragma unroll
      for (int h = 0; h < NDC; ++h) {
        uint32_t ov[kNR];
        tmem_ld16(tmem + lane_off + C::O_COL + kNR * h, ov);  // warp-collective
        tmem_wait_ld();
        const int d = 128 * h + t;
        if (d < D) {
#pragma unroll
          for (int q = 0; q < kNR; ++q) {
            if (q < M) {
              const float v = __uint_as_float(ov[q]);
              if (single) p.o[((size_t)bkv * M + q) * D + d] = v * fac[q];
              else p.part_o[(cb * M + q) * D + d] = v;
            }
          }
        }
      }
      if (t < M) {
        float mq = m_run[0], lq = l_tot[0], lsq = lse_row[0];
#pragma unroll
        for (int q = 1; q < kNR; ++q) {
          mq = (t == q) ? m_run[q] : mq;
          lq = (t == q) ? l_tot[q] : lq;
          lsq = (t == q) ? lse_row[q] : lsq;
        }
        if (single) {
          p.lse[(size_t)bkv * M + t] = lsq;
        } else {
          p.part_ml[(cb * M + t) * 2] = mq;
          p.part_ml[(cb * M + t) * 2 + 1] = lq;
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) atomicCAS(p.status, 0, kStatusTimeout);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// Merge of the chunks of one packed row (b * Hkv + kv head, m): with
// w_c = 2^(max_c - max), o = sum_c w_c O_c / sum_c w_c l_c and
// lse = (max + log2 sum_c w_c l_c) ln 2.  One block per row: the chunk
// weights are formed once in shared memory, then a thread per head-dim
// column sums its column over the chunks with independent loads.
constexpr int kMaxChunks = 1024;
__global__ void __launch_bounds__(128) decode_combine_kernel(DecParams p, int D) {
  __shared__ float wts[kMaxChunks];
  __shared__ float stat[2];
  const int row = blockIdx.x;  // (b * Hkv + kv head) * M + m
  const int rows = gridDim.x;
  const int nc = p.n_chunks;
  if (threadIdx.x < 32) {
    float mx = -INFINITY;
    for (int c = threadIdx.x; c < nc; c += 32) mx = fmaxf(mx, p.part_ml[((size_t)c * rows + row) * 2]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float l = 0.f;
    for (int c = threadIdx.x; c < nc; c += 32) {
      const float mc = p.part_ml[((size_t)c * rows + row) * 2];
      const float w = (mc == -INFINITY) ? 0.f : exp2f(mc - mx);  // a chunk that saw no key adds nothing
      wts[c] = w;
      l += w * p.part_ml[((size_t)c * rows + row) * 2 + 1];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (threadIdx.x == 0) {
      stat[0] = mx;
      stat[1] = l;
    }
  }
  __syncthreads();
  // 1 / l, or with attention sinks the factor that folds the row's head sink
  // into the normaliser (rows are (b Hkv + kv head) M + m, m = head-in-group
  // Lq + query row)
  float lse_out = (stat[0] + log2f(stat[1])) * kLn2;
  float inv = 1.f / stat[1];
  if (p.g.sinks) {
    const int bkv = row / p.M, m = row - bkv * p.M;
    inv = sink_finish(p.g.sinks[(bkv % p.g.Hkv) * p.g.G + m / p.g.Lq], stat[0], stat[1], &lse_out);
  }
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float t0 = 0.f, t1 = 0.f;
    int c = 0;
    for (; c + 1 < nc; c += 2) {
      t0 = fmaf(wts[c], p.part_o[((size_t)c * rows + row) * D + d], t0);
      t1 = fmaf(wts[c + 1], p.part_o[((size_t)(c + 1) * rows + row) * D + d], t1);
    }
    if (c < nc) t0 = fmaf(wts[c], p.part_o[((size_t)c * rows + row) * D + d], t0);
    p.o[(size_t)row * D + d] = (t0 + t1) * inv;
  }
  if (threadIdx.x == 0) p.lse[row] = lse_out;
}

// Key range of the group and its split into chunks of whole tiles, so that
// all CTAs run in one wave (at most 148 of the 152 SMs: the stream is bound
// by HBM, which that many SMs saturate, and one wave leaves no tail).
struct DecPlan {
  int k_begin, k_end, chunk, n_chunks;
};
DecPlan decode_plan(const Geom& g) {
  DecPlan pl;
  pl.k_begin = band_key_lo(g, 0);
  pl.k_end = band_key_hi(g, g.Lq - 1) + 1;
  const int KB = T;
  const int range = pl.k_end - pl.k_begin;
  const int groups = g.B * g.Hkv;
  int want = 148 / groups;
  const int max_chunks = (range + KB - 1) / KB;
  if (want > max_chunks) want = max_chunks;
  if (want < 1) want = 1;
  pl.chunk = ((range + want - 1) / want + KB - 1) / KB * KB;
  pl.n_chunks = (range + pl.chunk - 1) / pl.chunk;  // <= want <= 148, within the merge's kMaxChunks
  return pl;
}

template <int D>
cudaError_t decode_d(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v, float* o, float* lse,
                     float* ws, int* status, cudaStream_t s) {
  using C = DecCfg<D>;
  CUtensorMap tq, tk, tv;
  cudaError_t e;
  const int M = g.G * g.Lq;
  // q as [B * Hkv, M, D]: a 16-row box (rows past M read as zero); K and V in
  // slots of CPS 64-column chunks of 128 key rows, one TMA instruction each
  if ((e = make_tmap_f16(&tq, q, D, M, g.B * g.Hkv, kNR)) != cudaSuccess) return e;
  if ((e = make_tmap_f16_chunks(&tk, k, D, g.L, g.B * g.Hkv, T, C::CPS)) != cudaSuccess) return e;
  if ((e = make_tmap_f16_chunks(&tv, v, D, g.L, g.B * g.Hkv, T, C::CPS)) != cudaSuccess) return e;
  const DecPlan pl = decode_plan(g);
  DecParams p;
  p.g = g;
  p.o = o;
  p.lse = lse;
  p.M = M;
  p.k_begin = pl.k_begin;
  p.k_end = pl.k_end;
  p.chunk = pl.chunk;
  p.n_chunks = pl.n_chunks;
  p.part_o = ws;
  p.part_ml = ws + (size_t)pl.n_chunks * g.B * g.Hkv * M * D;
  p.status = status;
  auto kern = decode_kernel<D>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM)) != cudaSuccess)
    return e;
  kern<<<dim3(pl.n_chunks, g.B * g.Hkv), kThr, C::SMEM, s>>>(tq, tk, tv, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (pl.n_chunks > 1) {
    decode_combine_kernel<<<g.B * g.Hkv * M, 128, 0, s>>>(p, D);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace

bool decode_supported(const Geom& g) { return g.Rc == 0 && g.G * g.Lq <= kDecodeMaxRows; }

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
