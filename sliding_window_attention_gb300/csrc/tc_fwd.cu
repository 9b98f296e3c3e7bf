// Tensor-core forward for sm_103a: S = scale * Q K^T and O = P V on tcgen05
// with accumulators in Tensor Memory, operand tiles staged by TMA.
//
// One CTA per (128-row query tile, query head) -- and, at head dim 512, per
// 256-column half of O: O does not fit in TMEM whole, so each half-CTA
// recomputes S over the full head dim and accumulates its half.  Warp roles:
//   warp 0      TMA producer: Q once, then K and V tiles through an NS-deep ring
//   warp 1      TMEM allocation and the single-thread tcgen05.mma issuer
//   warps 2..   softmax: thread r of a warpgroup owns query row i0 + r (TMEM
//               lane r); reads its S row from TMEM, applies the band mask on
//               edge tiles, keeps the running max / sum, writes P (fp16) back
//               into the S columns for the TS-form PV MMA, rescales O when the
//               max grows, and writes O / l and lse at the end.  At head dim
//               <= 128 two warpgroups share every tile, 64 columns each (the
//               row max is combined through shared memory, the row sums are
//               kept per warpgroup in registers), which halves the softmax
//               latency that separates S(n) from PV(n); at larger head dims
//               one warpgroup takes whole tiles and the tensor core sums P
//               against a block of ones.
// The key tiles visited are exactly those that intersect the query tile's
// band ("Lab 028 lab detail: Off NVIDIA, you fix the platform yourself",
// "What I changed, in plain terms" item 3); inside edge tiles P is zeroed
// where j > i or i - j >= window (item 4).  The forward writes the row
// logsumexp the backward reuses (item 1).
//
// Operands are fp16 copies of the bf16 inputs (exact for |x| in [2^-14,
// 65504]): P is rounded to fp16 (11-bit significand) instead of bf16 for the
// PV product.  S and O accumulate in fp32.
//
// Rescaling is lazy: the running max used for P only moves when the tile max
// exceeds it by more than kRescaleLog2 (P values then stay <= 2^8, safe in
// fp16 and fp32); the final O / l is exact for any such choice.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "swa_internal.h"
#include "tc_ptx.cuh"

namespace swa {
namespace {

using namespace tc;

constexpr int kBM = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;

constexpr int kSmemMax = 232448;  // dynamic shared memory per block on sm_103 (227 KB)

template <int D>
struct FwdCfg {
  // key tile rows: the K (and V) tiles must leave room for >= 2 pipeline stages
  static constexpr int BN = 64;
  static constexpr int THREADS = 64 + 128;  // warp 0 TMA, warp 1 MMA, warps 2-5 softmax
  static constexpr int KCH = D / 64;                // 64-column (128-byte) chunks of a Q / K / V row
  static constexpr int Q_BYTES = kBM * D * 2;
  static constexpr int K_BYTES = BN * D * 2;
  static constexpr int V_BYTES = BN * D * 2;
  // mbarriers (512 B), then a block of ones (512 B)
  static constexpr int ONES_OFF = 512;
  static constexpr int BAR_BYTES = ONES_OFF + 512;
  // as many K/V stages as shared memory holds (TMA latency hiding), 2..8
  static constexpr int NS_FIT = (kSmemMax - 1024 - BAR_BYTES - Q_BYTES) / (K_BYTES + V_BYTES);
  static constexpr int NS = NS_FIT < 2 ? 2 : (NS_FIT > 8 ? 8 : NS_FIT);
  static constexpr int O_COL = 0;                   // O at [0, D)
  static constexpr int S_COL = 256;                 // S buffers at [256, 256 + 2 BN)
  // row sums l = P . 1 accumulated by the tensor core (16 identical columns)
  static constexpr int L_COL = S_COL + 2 * BN;
  static constexpr size_t SMEM = (size_t)Q_BYTES + (size_t)NS * (K_BYTES + V_BYTES) + BAR_BYTES + 1024 /*align*/;
  static_assert(SMEM <= (size_t)kSmemMax, "shared memory");
  static_assert(D == 256, "head dim 256 (64 and 128: fwd_pp_kernel; 512: the cluster kernel)");
  static_assert(S_COL + 2 * BN <= 512, "TMEM columns");
  static_assert(L_COL + 16 <= 512 && L_COL >= S_COL + 2 * BN, "TMEM columns for l");
};

struct FwdParams {
  Geom g;
  float* o;
  float* lse;
  int* status;
  int n_qtiles;
};

// One tile of the forward softmax for one row held in registers (raw scores
// sr[BN]): returns the tile's scaled row maximum through *tmax_out after
// pass 1; pass 2 (exp) runs in softmax_tile_p.  FULL: every entry is in the
// band (no masking code at all); otherwise entries outside the visible
// columns v (see vis(); TWO: two intervals, under a shared-prefix plan) are
// masked in the scaled domain, which is correct for any sign of the scale.
template <int BN, bool FULL, bool TWO = false>
__device__ __forceinline__ float softmax_tile_max(const uint32_t (&sr)[BN], float sl2, const int4& v) {
  float a0 = -INFINITY, a1 = -INFINITY;
  if constexpr (FULL) {
    if (sl2 >= 0.f) {
#pragma unroll
      for (int e = 0; e < BN; e += 4) {
        a0 = fmax3(a0, __uint_as_float(sr[e]), __uint_as_float(sr[e + 1]));
        a1 = fmax3(a1, __uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3]));
      }
      return fmaxf(a0, a1) * sl2;
    }
    float b0 = INFINITY, b1 = INFINITY, b2 = INFINITY, b3 = INFINITY;
#pragma unroll
    for (int e = 0; e < BN; e += 4) {
      b0 = fminf(b0, __uint_as_float(sr[e]));
      b1 = fminf(b1, __uint_as_float(sr[e + 1]));
      b2 = fminf(b2, __uint_as_float(sr[e + 2]));
      b3 = fminf(b3, __uint_as_float(sr[e + 3]));
    }
    return fminf(fminf(b0, b1), fminf(b2, b3)) * sl2;
  } else {
#pragma unroll
    for (int e = 0; e < BN; e += 2) {
      const float x0 = vis<TWO>(e, v) ? __uint_as_float(sr[e]) * sl2 : -INFINITY;
      const float x1 = vis<TWO>(e + 1, v) ? __uint_as_float(sr[e + 1]) * sl2 : -INFINITY;
      if (e & 2) a1 = fmaxf(a1, fmaxf(x0, x1));
      else a0 = fmaxf(a0, fmaxf(x0, x1));
    }
    return fmaxf(a0, a1);
  }
}

// Pass 2: P = 2^(sl2 * s - m) for the row, rounded to fp16, packed two per
// 32-bit TMEM column at p_taddr.  SUM: also returns the row sum of P (fp32);
// otherwise the tensor core takes it.  On full tiles the scaling and the two
// running sums use paired .f32x2 instructions (same roundings as scalar).
template <int BN, bool FULL, bool SUM, bool TWO = false>
__device__ __forceinline__ float softmax_tile_p(const uint32_t (&sr)[BN], float sl2, float m_use, const int4& v,
                                                 uint32_t p_taddr) {
  float s0 = 0.f, s1 = 0.f;
  const uint64_t sc2 = f2_pack(sl2, sl2), nm2 = f2_pack(-m_use, -m_use);
  uint64_t acc2 = f2_pack(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const int col = c * 32 + e;
      float p0, p1;
      if (FULL) {
        const float2 x = f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[col]), __uint_as_float(sr[col + 1])), sc2, nm2));
        p0 = fast_exp2(x.x);
        p1 = fast_exp2(x.y);
      } else {
        const float x0 = vis<TWO>(col, v) ? __uint_as_float(sr[col]) * sl2 : -INFINITY;
        const float x1 = vis<TWO>(col + 1, v) ? __uint_as_float(sr[col + 1]) * sl2 : -INFINITY;
        p0 = fast_exp2(x0 - m_use);
        p1 = fast_exp2(x1 - m_use);
      }
      if (SUM) {
        if (FULL) {
          acc2 = f2_add(acc2, f2_pack(p0, p1));
        } else {
          s0 += p0;
          s1 += p1;
        }
      }
      const __half2 hp = __floats2half2_rn(p0, p1);
      pk[e >> 1] = *reinterpret_cast<const uint32_t*>(&hp);
    }
    tmem_st16(p_taddr + c * 16, pk);
  }
  if (FULL) {
    const float2 t = f2_unpack(acc2);
    return t.x + t.y;
  }
  return s0 + s1;
}

// TWO: a shared-prefix plan is active (a row may see two key intervals); a
// separate instantiation keeps the plain kernel's code.
template <int D, bool TWO>
__global__ void __launch_bounds__(FwdCfg<D>::THREADS, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmO,  // fp32 o, 32 x 32 boxes
                  const FwdParams p) {
  using C = FwdCfg<D>;
  constexpr int BN = C::BN, NS = C::NS;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sQ = base;
  unsigned char* sK = sQ + C::Q_BYTES;
  unsigned char* sV = sK + NS * C::K_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + NS * C::V_BYTES);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + NS;
  uint64_t* v_full = k_empty + NS;
  uint64_t* v_empty = v_full + NS;
  uint64_t* s_full = v_empty + NS;  // [2]
  uint64_t* p_full = s_full + 2;    // [2]
  uint64_t* o_done = p_full + 2;    // [1]: PV into O complete
  uint64_t* mma_drain = o_done + 1;  // [1] every issued MMA finished (before TMEM is released)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // 16 x 16 block of fp16 ones (B operand of the row-sum MMA), no swizzle
  uint32_t* ones = reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(bars) + C::ONES_OFF);

  const Geom& g = p.g;
  const int warp = threadIdx.x / 32;
  const int bh = blockIdx.x;  // b * Hq + h
  const int b = bh / g.Hq, h = bh - b * g.Hq;
  const int bkv = b * g.Hkv + h / g.G;
  const int qt = p.n_qtiles - 1 - (int)blockIdx.y;  // longest rows first
  const int i0 = qt * kBM;
  const int ihi = min(i0 + kBM, g.Lq) - 1;
  // key tiles meeting the band of rows i0 .. ihi (never empty: every row
  // sees at least the key at its own position)
  const TileSteps steps = row_steps(g, i0, ihi, BN);
  const int nt = steps.count();
  constexpr bool two = TWO;  // shared-prefix plan: up to two visible intervals per row

  if (threadIdx.x < 128) ones[threadIdx.x] = 0x3C003C00u;  // two fp16 1.0 per word, 512 bytes
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(k_empty + s, 1);
      mbar_init(v_full + s, 1);
      mbar_init(v_empty + s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(s_full + s, 1);
      mbar_init(p_full + s, 128);
    }
    mbar_init(o_done, 1);
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // ones[] is read by the tensor core
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (elect_one()) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      mbar_arrive_expect_tx(q_full, C::Q_BYTES);
      tma_load_4d(sQ, &tmQ, q_full, 0, i0, 0, bh);  // all KCH chunks in one instruction
      int nk = 0, nv = 0;
      for (int n = 0; n < nt; ++n) {
        const int st = n % NS;
        const uint32_t par = ((n / NS) & 1) ^ 1;
        const int j0 = (two ? steps.tile(n) : steps.lo0 + n) * BN;
        if (n >= NS && !mbar_wait(k_empty + st, par, abort_flag)) break;
        mbar_arrive_expect_tx(k_full + st, C::K_BYTES);
        tma_load_4d(sK + st * C::K_BYTES, &tmK, k_full + st, 0, j0, 0, bkv);
        ++nk;
        if (n >= NS && !mbar_wait(v_empty + st, par, abort_flag)) break;
        mbar_arrive_expect_tx(v_full + st, C::V_BYTES);
        tma_load_4d(sV + st * C::V_BYTES, &tmV, v_full + st, 0, j0, 0, bkv);
        ++nv;
      }
      if (*abort_flag) {  // unwinding: the loads in flight land before shared memory is released
        mbar_wait_drain(q_full, 0);
        drain_ring(k_full, NS, nk);
        drain_ring(v_full, NS, nv);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (elect_one()) {
      const uint32_t idS = idesc_f16(kBM, BN, 1, 1, 0, 0);   // Q (K-major) x K (K-major), both bf16
      const uint32_t idPV = idesc_f16(kBM, D, 0, 0, 0, 1);   // P (TMEM) x V (MN-major)
      const uint32_t idL = idesc_f16(kBM, 16, 0, 0, 0, 0);   // P (TMEM) x ones (K-major)
      const uint64_t ones_desc = smem_desc_noswz(smem_u32(ones), 128, 256);
      const uint64_t qdesc = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      bool ok = mbar_wait(q_full, 0, abort_flag);
      auto issue_pv = [&](int m) -> bool {
        const int st = m % NS, sb = m & 1;
        if (!mbar_wait(p_full + sb, (m >> 1) & 1, abort_flag)) return false;
        if (!mbar_wait(v_full + st, (m / NS) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint64_t vdesc = smem_desc_sw128(smem_u32(sV + st * C::V_BYTES), BN * 128, 1024);
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks) {
          const uint64_t bdesc = desc_add(vdesc, ks * 2048);
          mma_ts(tmem + C::O_COL, tmem + C::S_COL + sb * BN + ks * 8, bdesc, idPV, (m > 0 || ks > 0) ? 1u : 0u);
        }
        // l += P . 1: every 16 x 16 step reads the same block of ones
        {
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks)
            mma_ts(tmem + C::L_COL, tmem + C::S_COL + sb * BN + ks * 8, ones_desc, idL, (m > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(o_done);
        mma_commit(v_empty + st);
        return true;
      };
      for (int n = 0; ok && n < nt; ++n) {
        const int st = n % NS, sb = n & 1;
        if (!mbar_wait(k_full + st, (n / NS) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint64_t kdesc = smem_desc_sw128(smem_u32(sK + st * C::K_BYTES), 16, 1024);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks & 3) * 32;  // 16 fp16 = 32 bytes along K inside a 128-byte chunk
          const uint64_t adesc = desc_add(qdesc, (ks >> 2) * kBM * 128 + off);
          const uint64_t bdesc = desc_add(kdesc, (ks >> 2) * BN * 128 + off);
          mma_ss(tmem + C::S_COL + sb * BN, adesc, bdesc, idS, ks > 0 ? 1u : 0u);
        }
        mma_commit(s_full + sb);
        mma_commit(k_empty + st);
        if (n >= 1 && !issue_pv(n - 1)) { ok = false; break; }
      }
      if (ok) issue_pv(nt - 1);
      // every MMA issued so far has finished before TMEM is released
      mma_commit(mma_drain);
      mbar_wait_drain(mma_drain, 0);
    }
  } else if (warp >= 2) {
    // ---------------- softmax / correction / epilogue (one warpgroup) ----------------
    const int r = 32 * (warp & 3) + (threadIdx.x & 31);
    const int i = i0 + r;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const float sl2 = g.scale * kLog2e;
    float m_run = -INFINITY;
    bool ok = true;
    // loop invariants: this row's band, and the bounds every row of the tile shares
    const int4 vrow = row_vis(g, i, 0);
    const int lo_all = band_key_lo(g, ihi), hi_all = band_key_hi(g, i0);
    for (int n = 0; n < nt; ++n) {
      const int sb = n & 1;
      const int j0 = (two ? steps.tile(n) : steps.lo0 + n) * BN;
      if (!__all_sync(0xffffffffu, mbar_wait(s_full + sb, (n >> 1) & 1, abort_flag))) { ok = false; break; }
      tc_fence_after();
      const bool full = two ? rows_tile_full(g, i0, ihi, j0, j0 + BN - 1) : (j0 >= lo_all && j0 + BN - 1 <= hi_all);
      // the whole S row in registers: all loads issued, then one wait
      uint32_t sr[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c)
        tmem_ld32(tmem + lane_off + C::S_COL + sb * BN + c * 32, *reinterpret_cast<uint32_t(*)[32]>(sr + c * 32));
      tmem_wait_ld();
      // Visible key columns of this row inside the tile (edge tiles only);
      // the two-interval mask only where a row of the warp needs it
      bool both = false;
      const int4 vv = two ? vis_in_tile(vshift(vrow, j0), BN, &both) : vshift(vrow, j0);
      const bool two_here = two && __any_sync(0xffffffffu, both);
      const float tmax = full ? softmax_tile_max<BN, true>(sr, sl2, vv)
                              : (two_here ? softmax_tile_max<BN, false, true>(sr, sl2, vv)
                                          : softmax_tile_max<BN, false>(sr, sl2, vv));
      float alpha = 1.f;
      bool rescale = false;
      if (tmax > m_run + kRescaleLog2) {
        if (m_run != -INFINITY) {
          alpha = fast_exp2(m_run - tmax);
          rescale = true;
        }
        m_run = tmax;
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      const uint32_t p_taddr = tmem + lane_off + C::S_COL + sb * BN;
      if (full) softmax_tile_p<BN, true, false>(sr, sl2, m_use, vv, p_taddr);
      else if (two_here) softmax_tile_p<BN, false, false, true>(sr, sl2, m_use, vv, p_taddr);
      else softmax_tile_p<BN, false, false>(sr, sl2, m_use, vv, p_taddr);
      // Wait for PV(n-1) at every tile, not only when rescaling: this thread then
      // has observed every earlier PV completion, so the o_done phase can be at
      // most one ahead of the parity asked for (no aliasing of phase n-3 with
      // n-1), and a rescale never overlaps an in-flight PV.
      if (n > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(o_done, (n - 1) & 1, abort_flag))) { ok = false; break; }
        tc_fence_after();
      }
      // tcgen05.ld/st are warp-collective: the whole warp rescales if any row needs it
      if (__any_sync(0xffffffffu, rescale) && n > 0) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(tmem + lane_off + C::O_COL + c * 32, rr);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
          tmem_st32(tmem + lane_off + C::O_COL + c * 32, rr);
        }
        {
          uint32_t lr[16];
          tmem_ld16(tmem + lane_off + C::L_COL, lr);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) lr[e] = __float_as_uint(__uint_as_float(lr[e]) * alpha);
          tmem_st16(tmem + lane_off + C::L_COL, lr);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full + sb);
    }
    // O and l are final once the last PV completes
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(o_done, (nt - 1) & 1, abort_flag));
    ok = __all_sync(0xffffffffu, ok && !*abort_flag);
    if (ok) {
      tc_fence_after();
      uint32_t lr[16];
      tmem_ld16(tmem + lane_off + C::L_COL, lr);  // warp-collective
      tmem_wait_ld();
      const float l_tot = __uint_as_float(lr[0]);
      const bool row_ok = i < g.Lq;
      // 1 / l, or with attention sinks the factor that folds the head's sink
      // logit into the row's normaliser
      float lse_row = (m_run + log2f(l_tot)) * kLn2;
      float inv = 1.f / l_tot;
      if (g.sinks) inv = sink_finish(g.sinks[bh % g.Hq], m_run, l_tot, &lse_row);
      // O through TMA stores, staged in 16 KB per warp of the (consumed) Q tile
      tmem_rows_store_tma(&tmO, tmem + lane_off + C::O_COL, 0, D, inv,
                          smem_u32(base) + (uint32_t)(warp - 2) * 16384u, i - (int)(threadIdx.x & 31), bh,
                          (int)(threadIdx.x & 31));
      if (row_ok) p.lse[(size_t)bh * g.Lq + i] = lse_row;
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

// ---------------------------------------------------------------------------
// bf16 -> fp16 operand copies (up to four tensors per launch; blockIdx.y
// selects the tensor).  Each thread moves two 16-byte vectors per iteration.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 in, bool& overflow) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float lo = __uint_as_float(w[e] << 16);
    const float hi = __uint_as_float(w[e] & 0xffff0000u);
    const __half2 hv = __floats2half2_rn(lo, hi);
    const float2 back = __half22float2(hv);
    overflow |= (isinf(back.x) && !isinf(lo)) || (isinf(back.y) && !isinf(hi));
    o[e] = *reinterpret_cast<const uint32_t*>(&hv);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// ===========================================================================
// Forward for head dims 64 and 128: two 128-row query tiles per CTA (rows
// 256 p .. 256 p + 255 of one head), each with its own softmax warpgroup, O
// accumulator and S buffer, sharing every K / V tile.  While one warpgroup
// turns its S into P, the tensor core works on the other tile, so the softmax
// of one tile hides behind the other's MMAs, and each K / V tile is read once
// for 256 query rows.
//
// TMEM: O of tile w at [w D, w D + D), S of tile w at [256 + 128 w, +128); P
// goes back as fp16 pairs into the first 64 columns of its S buffer.  Row
// sums stay in registers (a thread owns a whole row).  MMA issue order per key
// tile n: PV_A(n), S_A(n + 1), PV_B(n), S_B(n + 1): S_w(n + 1) overwrites
// P_w(n) only after PV_w(n) (one thread issues, the tensor pipe runs in
// order).  K and V travel in separate rings, filled by two producer lanes.
template <int D>
struct FwdPPCfg {
  static constexpr int BM = 128, BN = 128, KCH = D / 64;
  static constexpr int Q_BYTES = BM * D * 2;   // one query tile
  static constexpr int KV_BYTES = BN * D * 2;  // one K (or V) tile
  static constexpr int AVAIL = kSmemMax - 1024 /*align*/ - 1024 /*barriers*/ - 2 * Q_BYTES;
  static constexpr int NT = AVAIL / KV_BYTES;  // K and V tiles that fit
  static constexpr int NK = NT / 2 + NT % 2 > 6 ? 6 : NT / 2 + NT % 2;
  static constexpr int NV = NT / 2 > 6 ? 6 : NT / 2;
  static constexpr uint32_t S_COL = 256;
  static constexpr size_t SMEM = 2 * (size_t)Q_BYTES + (size_t)(NK + NV) * KV_BYTES + 1024 + 1024;
  static_assert(D == 64 || D == 128, "two O accumulators below the S buffers");
  static_assert(NK >= 2 && NV >= 2, "ring depth");
  static_assert(SMEM <= (size_t)kSmemMax, "shared memory");
};

// TWO: a shared-prefix plan is active (see fwd_tc_kernel).
template <int D, bool TWO>
__global__ void __launch_bounds__(352, 1)
    fwd_pp_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdPPCfg<D>;
  constexpr int BM = C::BM, BN = C::BN, NK = C::NK, NV = C::NV;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sQ = base;                    // [2][Q_BYTES]
  unsigned char* sK = sQ + 2 * C::Q_BYTES;     // [NK][KV_BYTES]
  unsigned char* sV = sK + NK * C::KV_BYTES;   // [NV][KV_BYTES]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + NV * C::KV_BYTES);
  uint64_t* q_full = bars;             // [1]
  uint64_t* k_full = q_full + 1;       // [NK]
  uint64_t* k_empty = k_full + NK;     // [NK]
  uint64_t* v_full = k_empty + NK;     // [NV]
  uint64_t* v_empty = v_full + NV;     // [NV]
  uint64_t* s_full = v_empty + NV;     // [2] S of tile w in TMEM
  uint64_t* p_full = s_full + 2;       // [2] P of tile w packed (and O rescaled) by its warpgroup
  uint64_t* o_done = p_full + 2;       // [2] PV of tile w finished
  uint64_t* mma_drain = o_done + 2;    // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const Geom& g = p.g;
  const int warp = threadIdx.x / 32;
  const int bh = blockIdx.x;  // b * Hq + h
  const int b = bh / g.Hq, h = bh - b * g.Hq;
  const int bkv = b * g.Hkv + h / g.G;
  const int pair = p.n_qtiles - 1 - (int)blockIdx.y;  // longest rows first (n_qtiles: pairs here)
  // tile w (A = 0, B = 1): query rows [i0w, ihiw]; its key tiles stA / stB
  // in ascending order (none when tile B has no rows).  Scalars, not arrays:
  // an array indexed by the warpgroup would live in local memory.
  const int i0A = 2 * pair * BM, i0B = i0A + BM;
  const int ihiA = min(i0A + BM, g.Lq) - 1, ihiB = min(i0B + BM, g.Lq) - 1;
  const TileSteps stA = row_steps(g, i0A, ihiA, BN);
  const TileSteps stB = i0B < g.Lq ? row_steps(g, i0B, ihiB, BN) : TileSteps{0, 0, 0, 0};
  const bool hasB = stB.count() > 0;
  constexpr bool two = TWO;  // shared-prefix plan: up to two visible intervals per row
  // (without a plan every query tile's key tiles are one range: part 0)
  auto first_tile = [](const TileSteps& s) { return (!two || s.n0) ? s.lo0 : s.lo1; };
  auto last_tile = [](const TileSteps& s) { return (two && s.n1) ? s.lo1 + s.n1 - 1 : s.lo0 + s.n0 - 1; };
  // key tiles of either query tile
  const int u0 = hasB ? min(first_tile(stA), first_tile(stB)) : first_tile(stA);
  const int u1 = hasB ? max(last_tile(stA), last_tile(stB)) : last_tile(stA);
  auto in_steps = [](const TileSteps& s, int n) {
    return (n >= s.lo0 && n < s.lo0 + s.n0) || (two && n >= s.lo1 && n < s.lo1 + s.n1);
  };
  auto uses = [&](int w, int n) { return w ? in_steps(stB, n) : in_steps(stA, n); };

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
    for (int w = 0; w < 2; ++w) {
      mbar_init(s_full + w, 1);
      mbar_init(p_full + w, 128);
      mbar_init(o_done + w, 1);
    }
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
    // ---------------------------------------------------------------- TMA producers
    // warp 0: both query tiles, then the K tiles; warp 10: the V tiles (a
    // warp of its own: two lanes of one warp spinning on different rings
    // delay each other).  Each stream is loaded in the order the MMA thread
    // consumes it (key tiles u0 .. u1 that either query tile uses) and waits
    // only on its own ring.
    const int lane = threadIdx.x & 31;
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      mbar_arrive_expect_tx(q_full, 2 * C::Q_BYTES);
      tma_load_4d(sQ, &tmQ, q_full, 0, i0A, 0, bh);
      tma_load_4d(sQ + C::Q_BYTES, &tmQ, q_full, 0, i0B, 0, bh);  // rows past Lq read as zero
      int nk = 0;
      for (int n = u0; n <= u1; ++n) {
        if (!uses(0, n) && !uses(1, n)) continue;
        const int s = nk % NK;
        if (nk >= NK && !mbar_wait(k_empty + s, ((nk / NK) & 1) ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(k_full + s, C::KV_BYTES);
        tma_load_4d(sK + s * C::KV_BYTES, &tmK, k_full + s, 0, n * BN, 0, bkv);
        ++nk;
      }
      if (*abort_flag) {  // unwinding: the loads in flight land before shared memory is released
        mbar_wait_drain(q_full, 0);
        drain_ring(k_full, NK, nk);
      }
    }
  } else if (warp == 10) {
    if ((threadIdx.x & 31) == 0) {
      int nv = 0;
      for (int n = u0; n <= u1; ++n) {
        if (!uses(0, n) && !uses(1, n)) continue;
        const int s = nv % NV;
        if (nv >= NV && !mbar_wait(v_empty + s, ((nv / NV) & 1) ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(v_full + s, C::KV_BYTES);
        tma_load_4d(sV + s * C::KV_BYTES, &tmV, v_full + s, 0, n * BN, 0, bkv);
        ++nv;
      }
      if (*abort_flag) drain_ring(v_full, NV, nv);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (elect_one()) {
      const uint32_t idS = idesc_f16(BM, BN, 1, 1, 0, 0);  // Q (K-major) x K (K-major), both bf16
      const uint32_t idPV = idesc_f16(BM, D, 0, 0, 0, 1);  // P (TMEM) x V (MN-major)
      int kc = 0, vc = 0;  // K / V tiles consumed
      int kpA = 0, kpB = 0;  // PV issued per query tile
      bool ok = mbar_wait(q_full, 0, abort_flag);
      // S_w from the K tile in slot kc % NK (waited for by the caller)
      auto issue_s = [&](int w) {
        const uint64_t qdesc = smem_desc_sw128(smem_u32(sQ + w * C::Q_BYTES), 16, 1024);
        const uint64_t kdesc = smem_desc_sw128(smem_u32(sK + (kc % NK) * C::KV_BYTES), 16, 1024);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks & 3) * 32;
          mma_ss(tmem + C::S_COL + 128 * w, desc_add(qdesc, (ks >> 2) * BM * 128 + off),
                 desc_add(kdesc, (ks >> 2) * BN * 128 + off), idS, ks > 0 ? 1u : 0u);
        }
        mma_commit(s_full + w);
      };
      auto wait_k = [&]() { return mbar_wait(k_full + kc % NK, (kc / NK) & 1, abort_flag); };
      // first key tile: S of each tile that uses it
      if (ok && (ok = wait_k())) {
        tc_fence_after();
        for (int w = 0; w < 2; ++w)
          if (uses(w, u0)) issue_s(w);
        mma_commit(k_empty + kc % NK);
        ++kc;
      }
      for (int n = u0; ok && n <= u1; ++n) {
        if (!uses(0, n) && !uses(1, n)) continue;
        int m = n + 1;  // the next key tile either query tile uses
        while (m <= u1 && !uses(0, m) && !uses(1, m)) ++m;
        const bool next = m <= u1;
        if (!mbar_wait(v_full + vc % NV, (vc / NV) & 1, abort_flag) || (next && !wait_k())) { ok = false; break; }
        tc_fence_after();
        const uint64_t vdesc = smem_desc_sw128(smem_u32(sV + (vc % NV) * C::KV_BYTES), BN * 128, 1024);
        for (int w = 0; w < 2 && ok; ++w) {
          if (uses(w, n)) {
            int& kp = w ? kpB : kpA;
            if (!mbar_wait(p_full + w, kp & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < BN / 16; ++ks)
              mma_ts(tmem + D * w, tmem + C::S_COL + 128 * w + ks * 8, desc_add(vdesc, ks * 2048), idPV,
                     (kp > 0 || ks > 0) ? 1u : 0u);
            mma_commit(o_done + w);
            ++kp;
          }
          if (next && uses(w, m)) issue_s(w);  // after PV_w(n): S_w(m) overwrites P_w(n)
        }
        if (!ok) break;
        mma_commit(v_empty + vc % NV);
        ++vc;
        if (next) {
          mma_commit(k_empty + kc % NK);
          ++kc;
        }
      }
      // every MMA issued so far has finished before TMEM is released
      mma_commit(mma_drain);
      mbar_wait_drain(mma_drain, 0);
    }
  } else {
    // ---------------------------------------------------------------- softmax, one warpgroup per query tile
    const int w = (warp - 2) >> 2;  // warps 2-5: tile A, 6-9: tile B
    const int r = 32 * (warp & 3) + (threadIdx.x & 31);
    const int i0w = w ? i0B : i0A, ihiw = w ? ihiB : ihiA;
    const TileSteps stw = w ? stB : stA;
    const int i = i0w + r;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t s_col = C::S_COL + 128 * w, o_col = D * w;
    const float sl2 = g.scale * kLog2e;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    const int cnt = stw.count();  // key tiles of this query tile (0 for a missing tile B)
    const int4 vrow = row_vis(g, i, 0);
    const int lo_all = band_key_lo(g, ihiw), hi_all = band_key_hi(g, i0w);
    for (int k = 0; k < cnt; ++k) {
      const int j0 = (two ? stw.tile(k) : stw.lo0 + k) * BN;
      if (!__all_sync(0xffffffffu, mbar_wait(s_full + w, k & 1, abort_flag))) { ok = false; break; }
      tc_fence_after();
      const bool full = two ? rows_tile_full(g, i0w, ihiw, j0, j0 + BN - 1)
                            : (j0 >= lo_all && j0 + BN - 1 <= hi_all);
      const int4 vv = vshift(vrow, j0);
      // the row in two 64-column halves (registers stay below the spill
      // limit): first the maximum, then P; half h's packed P lands on columns
      // [32 h, 32 h + 32), which half h has already read
      float tmax = -INFINITY;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t sr[64];
        tmem_ld32(tmem + lane_off + s_col + 64 * hf, *reinterpret_cast<uint32_t(*)[32]>(sr));
        tmem_ld32(tmem + lane_off + s_col + 64 * hf + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
        tmem_wait_ld();
        bool both = false;
        const int4 vh = two ? vis_in_tile(vshift(vv, 64 * hf), 64, &both) : vshift(vv, 64 * hf);
        const bool two_here = two && __any_sync(0xffffffffu, both);
        tmax = fmaxf(tmax, full ? softmax_tile_max<64, true>(sr, sl2, vh)
                                : (two_here ? softmax_tile_max<64, false, true>(sr, sl2, vh)
                                            : softmax_tile_max<64, false>(sr, sl2, vh)));
      }
      float alpha = 1.f;
      bool rescale = false;
      if (tmax > m_run + kRescaleLog2) {
        if (m_run != -INFINITY) {
          alpha = fast_exp2(m_run - tmax);
          rescale = true;
        }
        m_run = tmax;
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      float tsum = 0.f;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t sr[64];
        tmem_ld32(tmem + lane_off + s_col + 64 * hf, *reinterpret_cast<uint32_t(*)[32]>(sr));
        tmem_ld32(tmem + lane_off + s_col + 64 * hf + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
        tmem_wait_ld();
        const uint32_t p_taddr = tmem + lane_off + s_col + 32 * hf;
        bool both = false;
        const int4 vh = two ? vis_in_tile(vshift(vv, 64 * hf), 64, &both) : vshift(vv, 64 * hf);
        const bool two_here = two && __any_sync(0xffffffffu, both);
        tsum += full ? softmax_tile_p<64, true, true>(sr, sl2, m_use, vh, p_taddr)
                     : (two_here ? softmax_tile_p<64, false, true, true>(sr, sl2, m_use, vh, p_taddr)
                                 : softmax_tile_p<64, false, true>(sr, sl2, m_use, vh, p_taddr));
      }
      l_run = l_run * alpha + tsum;
      // PV_w(k - 1) must be complete before O is rescaled (waited for at every
      // tile, so the o_done phase never runs more than one ahead)
      if (k > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(o_done + w, (k - 1) & 1, abort_flag))) { ok = false; break; }
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, rescale) && k > 0) {  // tcgen05.ld/st are warp-collective
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(tmem + lane_off + o_col + c * 32, rr);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
          tmem_st32(tmem + lane_off + o_col + c * 32, rr);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full + w);
    }
    if (ok && cnt > 0) ok = __all_sync(0xffffffffu, mbar_wait(o_done + w, (cnt - 1) & 1, abort_flag));
    ok = __all_sync(0xffffffffu, ok && !*abort_flag);
    if (ok && cnt > 0) {
      tc_fence_after();
      const bool row_ok = i < g.Lq;
      // 1 / l, or with attention sinks the factor that folds the head's sink
      // logit into the row's normaliser
      float lse_row = (m_run + log2f(l_run)) * kLn2;
      float inv = 1.f / l_run;
      if (g.sinks) inv = sink_finish(g.sinks[bh % g.Hq], m_run, l_run, &lse_row);
      // (row stores: at D <= 128 a warp's own quarter of its Q tile holds at
      // most two 4 KB staging buffers, and TMA stores through them measured
      // about 1% slower here)
      float* orow = p.o + ((size_t)bh * g.Lq + (row_ok ? i : 0)) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t acc[32];
        tmem_ld32(tmem + lane_off + o_col + c * 32, acc);
        tmem_wait_ld();  // warp-collective: every lane loads, only valid rows store
        if (row_ok) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(orow + c * 32 + e) =
                make_float4(__uint_as_float(acc[e]) * inv, __uint_as_float(acc[e + 1]) * inv,
                            __uint_as_float(acc[e + 2]) * inv, __uint_as_float(acc[e + 3]) * inv);
        }
      }
      if (row_ok) p.lse[(size_t)bh * g.Lq + i] = lse_row;
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

__global__ void __launch_bounds__(256) convert_bf16_f16_kernel(const uint16_t* s0, uint16_t* d0, long long n0,
                                                               const uint16_t* s1, uint16_t* d1, long long n1,
                                                               const uint16_t* s2, uint16_t* d2, long long n2,
                                                               const uint16_t* s3, uint16_t* d3, long long n3,
                                                               int* status, int* zero_word) {
  if (zero_word && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *zero_word = 0;
  const int seg = blockIdx.y;
  const uint4* src = reinterpret_cast<const uint4*>(seg == 0 ? s0 : seg == 1 ? s1 : seg == 2 ? s2 : s3);
  uint4* dst = reinterpret_cast<uint4*>(seg == 0 ? d0 : seg == 1 ? d1 : seg == 2 ? d2 : d3);
  const long long n16 = (seg == 0 ? n0 : seg == 1 ? n1 : seg == 2 ? n2 : n3) / 8;  // 16-byte vectors
  bool overflow = false;
  const long long stride = (long long)gridDim.x * blockDim.x;
  long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  // four 16-byte vectors in flight per thread
  for (; idx + 3 * stride < n16; idx += 4 * stride) {
    const uint4 a = __ldcs(src + idx);
    const uint4 b = __ldcs(src + idx + stride);
    const uint4 c = __ldcs(src + idx + 2 * stride);
    const uint4 d = __ldcs(src + idx + 3 * stride);
    dst[idx] = bf16x8_to_f16x8(a, overflow);
    dst[idx + stride] = bf16x8_to_f16x8(b, overflow);
    dst[idx + 2 * stride] = bf16x8_to_f16x8(c, overflow);
    dst[idx + 3 * stride] = bf16x8_to_f16x8(d, overflow);
  }
  for (; idx < n16; idx += stride) dst[idx] = bf16x8_to_f16x8(__ldcs(src + idx), overflow);
  if (overflow) atomicCAS(status, 0, kStatusFp16Range);
}

// ---------------------------------------------------------------------------
// Self-test of the device-side timeout path: one thread waits on an mbarrier
// that nothing arrives on, with a short cycle limit, through the same bounded
// wait every kernel uses, and latches the timeout in the status word.
__global__ void __launch_bounds__(32) selftest_timeout_kernel(int* status, long long limit_cycles) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0 && !mbar_wait_limit(&bar, 0, &abort_flag, limit_cycles)) atomicCAS(status, 0, kStatusTimeout);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

}  // namespace

cudaError_t launch_selftest_timeout(int* status, long long limit_cycles, cudaStream_t s) {
  selftest_timeout_kernel<<<1, 32, 0, s>>>(status, limit_cycles);
  return cudaGetLastError();
}

// 3-D fp16 tensor map over [heads, L, D] with a (64 x rows) box, 128-byte swizzle.
cudaError_t make_tmap_f16(CUtensorMap* m, const void* ptr, int D, int L, int heads, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L, (cuuint64_t)heads};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)D * L * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 4-D view (64 elements, L rows, D / 64 chunks, heads) of the same fp16
// [heads, L, D] tensor: one box (64, box_rows, nchunk, 1) lands as nchunk
// consecutive [box_rows x 128 B] swizzled blocks -- the layout of nchunk
// separate 3-D boxes -- in a single TMA instruction.  Measured on GB300, one
// 32 KB instruction sustains about 81 B/clk per SM against 67 for two 16 KB
// instructions under one barrier (46 for one 16 KB instruction).
cudaError_t make_tmap_f16_chunks(CUtensorMap* m, const void* ptr, int D, int L, int heads, int box_rows,
                                 int nchunk) {
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  if (nchunk < 1 || nchunk > D / 64) return cudaErrorInvalidValue;
  cuuint64_t dims[4] = {64, (cuuint64_t)L, (cuuint64_t)(D / 64), (cuuint64_t)heads};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, 128, (cuuint64_t)D * L * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)box_rows, (cuuint32_t)nchunk, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_f32_out(CUtensorMap* m, void* ptr, int D, int L, int heads) {
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  if (D % 32) return cudaErrorInvalidValue;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L, (cuuint64_t)heads};
  cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)D * L * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_convert_f16(const uint16_t* const* src, uint16_t* const* dst, const size_t* n, int count,
                               int* status, cudaStream_t s, int* zero_word) {
  if (count < 1 || count > 4) return cudaErrorInvalidValue;
  const uint16_t* sp[4] = {nullptr, nullptr, nullptr, nullptr};
  uint16_t* dp[4] = {nullptr, nullptr, nullptr, nullptr};
  long long nn[4] = {0, 0, 0, 0};
  long long most = 0;
  for (int i = 0; i < count; ++i) {
    sp[i] = src[i];
    dp[i] = dst[i];
    nn[i] = (long long)n[i];
    most = nn[i] > most ? nn[i] : most;
  }
  // blocks per tensor: enough for ~8 resident blocks per SM over all tensors
  long long blocks = (most / 8 + 511) / 512;
  const long long cap = (152LL * 8 + count - 1) / count;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  dim3 grid((unsigned)blocks, count);
  convert_bf16_f16_kernel<<<grid, 256, 0, s>>>(sp[0], dp[0], nn[0], sp[1], dp[1], nn[1], sp[2], dp[2], nn[2], sp[3],
                                              dp[3], nn[3], status, zero_word);
  return cudaGetLastError();
}

template <int D>
static cudaError_t fwd_tc_d(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v16, float* o,
                            float* lse, int* status, cudaStream_t s) {
  using C = FwdCfg<D>;
  CUtensorMap tq, tk, tv;
  cudaError_t e;
  // one TMA instruction per tile: Q, K and V in all D / 64 chunks
  if ((e = make_tmap_f16_chunks(&tq, q, D, g.Lq, g.B * g.Hq, kBM, C::KCH)) != cudaSuccess) return e;
  if ((e = make_tmap_f16_chunks(&tk, k, D, g.L, g.B * g.Hkv, C::BN, C::KCH)) != cudaSuccess) return e;
  if ((e = make_tmap_f16_chunks(&tv, v16, D, g.L, g.B * g.Hkv, C::BN, C::KCH)) != cudaSuccess) return e;
  auto kern = g.Rc > 0 ? fwd_tc_kernel<D, true> : fwd_tc_kernel<D, false>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM)) != cudaSuccess)
    return e;
  FwdParams p;
  p.g = g;
  p.o = o;
  p.lse = lse;
  p.status = status;
  p.n_qtiles = (g.Lq + kBM - 1) / kBM;
  dim3 grid(g.B * g.Hq, p.n_qtiles);
  CUtensorMap to;
  if ((e = make_tmap_f32_out(&to, o, D, g.Lq, g.B * g.Hq)) != cudaSuccess) return e;
  kern<<<grid, C::THREADS, C::SMEM, s>>>(tq, tk, tv, to, p);
  return cudaGetLastError();
}

template <int D>
static cudaError_t fwd_pp_d(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v16, float* o,
                            float* lse, int* status, cudaStream_t s) {
  using C = FwdPPCfg<D>;
  CUtensorMap tq, tk, tv;
  cudaError_t e;
  // one TMA instruction per tile: all D / 64 chunks
  if ((e = make_tmap_f16_chunks(&tq, q, D, g.Lq, g.B * g.Hq, C::BM, C::KCH)) != cudaSuccess) return e;
  if ((e = make_tmap_f16_chunks(&tk, k, D, g.L, g.B * g.Hkv, C::BN, C::KCH)) != cudaSuccess) return e;
  if ((e = make_tmap_f16_chunks(&tv, v16, D, g.L, g.B * g.Hkv, C::BN, C::KCH)) != cudaSuccess) return e;
  auto kern = g.Rc > 0 ? fwd_pp_kernel<D, true> : fwd_pp_kernel<D, false>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM)) != cudaSuccess)
    return e;
  FwdParams p;
  p.g = g;
  p.o = o;
  p.lse = lse;
  p.status = status;
  const int n_qtiles = (g.Lq + C::BM - 1) / C::BM;
  p.n_qtiles = (n_qtiles + 1) / 2;  // pairs of query tiles
  dim3 grid(g.B * g.Hq, p.n_qtiles);
  kern<<<grid, 352, C::SMEM, s>>>(tq, tk, tv, p);  // warps 0-9 and the V producer (warp 10)
  return cudaGetLastError();
}

bool fwd_tc_supported(int D) { return D == 64 || D == 128 || D == 256 || D == 512; }

cudaError_t launch_fwd_tc(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v16, float* o,
                          float* lse, int* work, int* status, cudaStream_t s) {
  switch (g.D) {
    case 64: return fwd_pp_d<64>(g, q, k, v16, o, lse, status, s);
    case 128: return fwd_pp_d<128>(g, q, k, v16, o, lse, status, s);
    case 256: return fwd_tc_d<256>(g, q, k, v16, o, lse, status, s);
    case 512: return launch_fwd_tc512(g, q, k, v16, o, lse, work, status, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace swa
