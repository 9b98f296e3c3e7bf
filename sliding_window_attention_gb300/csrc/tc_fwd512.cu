// Tensor-core forward for head dim 512 on 2-CTA thread-block clusters.
//
// At D = 512 the output accumulator O of a 128-row query tile (512 fp32
// columns) fills one SM's Tensor Memory, so S and O cannot live on the same
// SM.  One cluster per (query head, 128-row query tile), longest rows first:
//   rank 0 (producer): Q sits in Tensor Memory as fp16 pairs (256 columns,
//     the A operand of TS-form MMAs); K streams in 128-column slices, one
//     32 KB TMA instruction each (the per-SM TMA rate grows with the size of
//     an instruction: about 46 B/clk for 16 KB, 81 for 32 KB);
//     S = Q K^T (N = 128) into two TMEM buffers; online softmax with the band
//     mask on edge tiles ("Lab 028 lab detail: Off NVIDIA, you fix the
//     platform yourself", "What I changed, in plain terms" items 3-4); P in
//     fp16 is staged and bulk-copied into the accumulator's operand slot with
//     the per-row factor by which O must be rescaled; at the end it writes
//     the row logsumexp (same section, item 1) and sends 1 / l.
//   rank 1 (accumulator): O (512 columns) in Tensor Memory; V streams in
//     128-column chunks; before O += P V of a step its elementwise warps
//     rescale the rows whose running maximum moved (the maximum moves lazily,
//     only when it grows by more than 2^8, so this is rare); at the end it
//     writes O / l.
// Each side issues 2048 MMA cycles per 128 x 128 step and one 32 KB tile
// crosses distributed shared memory per step.
//
// Warps: 0 TMA, 1 TMEM owner and MMA issuer, 2-9 elementwise (two
// warpgroups, 64 columns of S or 256 columns of O each), 10 slot release
// (accumulator).  Every wait is bounded; a timeout in one CTA is broadcast to
// the cluster, every CTA drains its loads, copies and MMAs, and the status
// word records it.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "swa_internal.h"
#include "tc_ptx.cuh"

namespace swa {
namespace {

using namespace tc;

constexpr int T = 128;     // query rows per tile and key rows per step
constexpr int DH = 512;    // head dim
constexpr int kThr = 352;  // 11 warps
constexpr int kSigWarp = 10;
constexpr uint32_t R = 2;  // CTAs per cluster
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;

constexpr int TILE_BYTES = T * T * 2;       // fp16 128 x 128 P tile
constexpr int HALF_BYTES = TILE_BYTES / 2;  // one warpgroup's 64 columns (one swizzle chunk)
// producer shared memory: two staging tiles (P of step n goes to tile n % 2,
// so its copy is in flight while the next step's P is formed), row vectors,
// K ring
constexpr int OFF_STG = 0;
constexpr int OFF_VEC = 2 * TILE_BYTES;  // alpha[2][128], inv_l[128], max exchange [2][2][128], l exchange [2][128]
constexpr int OFF_RING_P = OFF_VEC + 8192;  // 1 KB aligned
constexpr int SLOT_P = T * 128 * 2;      // 128-column K slice: two TMA boxes under one barrier
constexpr int NR_P = 4;
// accumulator shared memory: two P slots, two alpha slots + 1 / l, V ring
constexpr int OFF_RECV = 0;
constexpr int OFF_RVEC = 2 * TILE_BYTES;  // alpha slot [2][128], inv_l [128]
constexpr int OFF_RING_A = 2 * TILE_BYTES + 2048;
constexpr int SLOT_A = T * 128 * 2;       // 128-column V chunk
constexpr int NR_A = 4;
constexpr int DATA_P = OFF_RING_P + NR_P * SLOT_P;
constexpr int DATA_A = OFF_RING_A + NR_A * SLOT_A;
constexpr int DATA_BYTES = DATA_P > DATA_A ? DATA_P : DATA_A;
constexpr uint32_t X_COL = 0, S_COL = 256;  // producer TMEM: Q [0, 256), S buffers [256, 512)
static_assert(OFF_VEC + 1024 + 512 + 2048 + 1024 <= OFF_RING_P, "producer vectors");
static_assert(OFF_RING_A % 1024 == 0 && OFF_RING_P % 1024 == 0, "swizzled tiles need 1 KB alignment");

struct Bars {
  uint64_t ring_full[11], ring_empty[11];
  uint64_t q_ready;                   // (producer) Q in TMEM
  uint64_t s_full[2], s_free[2];      // (producer) S buffers
  uint64_t mx[2];                     // (producer) both warpgroups posted their partial row max
  uint64_t staged[2];                 // (producer) a warpgroup wrote its staging half
  uint64_t stg_free[2][2];            // (producer) the copy out of staging half [tile][warpgroup] landed
  uint64_t dst_free[2];               // (producer) accumulator slot may be written
  uint64_t lx;                        // (producer) both warpgroups posted their row sums
  uint64_t fin_staged;                // (producer) 1 / l written
  uint64_t recv_full[2];              // (accumulator) P tile + alpha landed
  uint64_t o_ready[2];                // (accumulator) O rescaled for the step
  uint64_t mma_done[2];               // (accumulator) PV of a step finished
  uint64_t fin_full;                  // (accumulator) 1 / l landed
  uint64_t acc_done, mma_drain;
  uint32_t tmem_slot;
  int abort_flag;
  int n_sent[2];                      // (producer) steps copied, per warpgroup
  int fin_sent;
  int n_recv;                         // (accumulator) steps received
};
static_assert(NR_P <= 11 && NR_A <= 11, "ring barriers");

constexpr size_t SMEM = (size_t)DATA_BYTES + 1024 + 1024;
static_assert(SMEM <= 232448, "shared memory");
static_assert(sizeof(Bars) <= 1024, "barrier block");

struct FwdParams512 {
  Geom g;
  const uint16_t* q;  // bf16: S = Q K^T reads the caller's q and k as they are
  float* o;
  float* lse;
  int n_tiles;
  int* status;
};

// Scaled maximum over 64 raw scores of one row; entries outside [clo, chi]
// are excluded unless FULL (correct for any sign of the scale).
template <bool FULL>
__device__ __forceinline__ float half_max(const uint32_t (&sr)[64], float sl2, int clo, int chi) {
  float a0 = -INFINITY, a1 = -INFINITY;
#pragma unroll
  for (int e = 0; e < 64; e += 2) {
    float x0 = __uint_as_float(sr[e]) * sl2, x1 = __uint_as_float(sr[e + 1]) * sl2;
    if (!FULL) {
      x0 = (e >= clo && e <= chi) ? x0 : -INFINITY;
      x1 = (e + 1 >= clo && e + 1 <= chi) ? x1 : -INFINITY;
    }
    a0 = fmaxf(a0, x0);
    a1 = fmaxf(a1, x1);
  }
  return fmaxf(a0, a1);
}

// P = 2^(sl2 s - m) for 64 entries as fp16 pairs; returns the fp32 row sum.
template <bool FULL>
__device__ __forceinline__ float half_p(const uint32_t (&sr)[64], float sl2, float m_use, int clo, int chi,
                                        uint32_t (&pk)[32]) {
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int e = 0; e < 64; e += 2) {
    float p0 = fast_exp2(fmaf(__uint_as_float(sr[e]), sl2, -m_use));
    float p1 = fast_exp2(fmaf(__uint_as_float(sr[e + 1]), sl2, -m_use));
    if (!FULL) {
      p0 = (e >= clo && e <= chi) ? p0 : 0.f;
      p1 = (e + 1 >= clo && e + 1 <= chi) ? p1 : 0.f;
    }
    s0 += p0;
    s1 += p1;
    pk[e >> 1] = pack_half2(p0, p1);
  }
  return s0 + s1;
}

__global__ void __launch_bounds__(kThr, 1)
    fwd512_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const FwdParams512 p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(base + DATA_BYTES);
  volatile int* abort_flag = &bars->abort_flag;
  const uint32_t sbase = smem_u32(base);

  const Geom& g = p.g;
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool producer = rank == 0;
  // Grid (x, y, z) = (2 x the group's query heads, query tiles, b * Hkv + kv
  // head).  Blocks launch x fastest and z slowest, so the clusters running at
  // any moment share one kv head, whose K and V then stay in L2.
  const int bkv = (int)blockIdx.z;
  const int b = bkv / g.Hkv;
  const int bh = b * g.Hq + (bkv - b * g.Hkv) * g.G + (int)(blockIdx.x / R);  // b * Hq + query head
  const int tile = p.n_tiles - 1 - (int)blockIdx.y;  // longest rows first
  const int i0 = tile * T;
  const int ihi = min(i0 + T, g.Lq) - 1;
  const int t_lo = band_key_lo(g, i0) / T;
  const int N = band_key_hi(g, ihi) / T - t_lo + 1;  // key steps (at least one)

  if (threadIdx.x == 0) {
    for (int s = 0; s < 11; ++s) {
      mbar_init(&bars->ring_full[s], 1);
      mbar_init(&bars->ring_empty[s], 1);
    }
    mbar_init(&bars->q_ready, 256);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->s_free[s], 256);
      mbar_init(&bars->mx[s], 256);
      mbar_init(&bars->staged[s], 128);
      mbar_init(&bars->stg_free[s][0], 1);
      mbar_init(&bars->stg_free[s][1], 1);
      mbar_init(&bars->dst_free[s], 1);
      mbar_init(&bars->recv_full[s], 1);
      mbar_init(&bars->o_ready[s], 256);
      mbar_init(&bars->mma_done[s], 1);
      bars->n_sent[s] = 0;
    }
    mbar_init(&bars->lx, 256);
    mbar_init(&bars->fin_staged, 128);
    mbar_init(&bars->fin_full, 1);
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->mma_drain, 1);
    bars->abort_flag = 0;
    bars->fin_sent = 0;
    bars->n_recv = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // every CTA's barriers exist before any remote arrive or copy
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one()) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      int issued = 0;
      bool ok = true;
      const int nr = producer ? NR_P : NR_A;
      for (int n = 0; ok && n < N; ++n) {
        const int j0 = (t_lo + n) * T;
        for (int c = 0; c < DH / 128; ++c, ++issued) {
          const int s = issued % nr;
          if (issued >= nr && !mbar_wait_cl(&bars->ring_empty[s], ((issued / nr) & 1) ^ 1, abort_flag, R)) {
            ok = false;
            break;
          }
          if (producer) {
            unsigned char* dst = base + OFF_RING_P + s * SLOT_P;
            mbar_arrive_expect_tx(&bars->ring_full[s], SLOT_P);
            tma_load_4d(dst, &tmK, &bars->ring_full[s], 0, j0, 2 * c, bkv);  // chunks 2c, 2c + 1
          } else {
            unsigned char* dst = base + OFF_RING_A + s * SLOT_A;
            mbar_arrive_expect_tx(&bars->ring_full[s], SLOT_A);
            tma_load_4d(dst, &tmV, &bars->ring_full[s], 0, j0, 2 * c, bkv);
          }
        }
      }
      if (!ok) {
        // unwinding: let the loads in flight land (at most one per slot)
        for (int k = issued - 1; k >= 0 && k >= issued - nr; --k)
          mbar_wait_drain(&bars->ring_full[k % nr], (k / nr) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      bool ok = true;
      const uint32_t idS = idesc_f16(T, T, 1, 1, 0, 0);     // Q (TMEM) x K slice (K-major), both bf16
      const uint32_t idPV = idesc_f16(T, 128, 0, 0, 0, 1);  // P (K-major) x V chunk (MN-major)
      int used = 0;
      if (producer) {
        ok = mbar_wait_cl(&bars->q_ready, 0, abort_flag, R);
        for (int n = 0; ok && n < N; ++n) {
          const int bb = n & 1;
          if (n >= 2 && !mbar_wait_cl(&bars->s_free[bb], ((n >> 1) & 1) ^ 1, abort_flag, R)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int c = 0; c < DH / 128; ++c, ++used) {
            const int s = used % NR_P;
            if (!mbar_wait_cl(&bars->ring_full[s], (used / NR_P) & 1, abort_flag, R)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t kd = smem_desc_sw128(sbase + OFF_RING_P + s * SLOT_P, 16, 1024);
            // head-dim columns [128 c, 128 c + 128): Q columns 64 c + 8 ks in TMEM
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              mma_ts(tmem + S_COL + bb * T, tmem + X_COL + c * 64 + ks * 8,
                     desc_add(kd, (ks >> 2) * T * 128 + (ks & 3) * 32), idS, (c | ks) ? 1u : 0u);
            mma_commit(&bars->ring_empty[s]);
          }
          if (!ok) break;
          mma_commit(&bars->s_full[bb]);
        }
      } else {
        for (int n = 0; ok && n < N; ++n) {
          const int bb = n & 1;
          if (!mbar_wait_cl(&bars->o_ready[bb], (n >> 1) & 1, abort_flag, R)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = smem_desc_sw128(sbase + OFF_RECV + bb * TILE_BYTES, 16, 1024);
          for (int c = 0; c < DH / 128; ++c, ++used) {
            const int s = used % NR_A;
            if (!mbar_wait_cl(&bars->ring_full[s], (used / NR_A) & 1, abort_flag, R)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t vd = smem_desc_sw128(sbase + OFF_RING_A + s * SLOT_A, T * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < T / 16; ++ks)
              mma_ss(tmem + c * 128, desc_add(ad, (ks >> 2) * T * 128 + (ks & 3) * 32), desc_add(vd, ks * 2048),
                     idPV, (n | ks) ? 1u : 0u);
            mma_commit(&bars->ring_empty[s]);
          }
          if (!ok) break;
          mma_commit(&bars->mma_done[bb]);
        }
        if (ok) mma_commit(&bars->acc_done);
      }
      // every MMA issued so far has finished before TMEM is released
      mma_commit(&bars->mma_drain);
      mbar_wait_drain(&bars->mma_drain, 0);
    }
  } else if (warp == kSigWarp) {
    // ------------------------------------------------------------ slot release (accumulator)
    if (!producer && elect_one()) {
      mbar_arrive_expect_tx(&bars->fin_full, 512);
      for (int s = 0; s < 2 && s < N; ++s) {
        mbar_arrive_expect_tx(&bars->recv_full[s], TILE_BYTES + 512);
        mbar_arrive_remote(mapa(smem_u32(&bars->dst_free[s]), 0));
      }
      for (int n = 0; n + 2 < N; ++n) {
        if (!mbar_wait_cl(&bars->mma_done[n & 1], (n >> 1) & 1, abort_flag, R)) break;
        mbar_arrive_expect_tx(&bars->recv_full[n & 1], TILE_BYTES + 512);
        mbar_arrive_remote(mapa(smem_u32(&bars->dst_free[n & 1]), 0));
      }
    }
  } else if (producer) {
    // ------------------------------------------------------------ softmax (producer)
    const int wg = (warp - 2) >> 2, q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const int i = i0 + r;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const int cb0 = 64 * wg;
    const float sl2 = g.scale * kLog2e;
    float* alph = reinterpret_cast<float*>(base + OFF_VEC);  // [2 tile][128]
    float* finl = alph + 256;                                 // [128]
    float* xm = finl + 128;                                   // [2 parity][2 wg][128]
    float* xl = xm + 512;                                     // [2 wg][128]
    {
      // Q row i into Tensor Memory: fp16 pairs, one 32-bit column each; warpgroup
      // wg fills columns [128 wg, 128 wg + 128) (head-dim elements [256 wg, 256 wg + 256))
      const uint4* src =
          reinterpret_cast<const uint4*>(p.q + ((size_t)bh * g.Lq + (i < g.Lq ? i : 0)) * DH) + wg * 32;
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        uint32_t v[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 w4 = i < g.Lq ? __ldg(src + j * 8 + q) : make_uint4(0u, 0u, 0u, 0u);
          v[4 * q] = w4.x;
          v[4 * q + 1] = w4.y;
          v[4 * q + 2] = w4.z;
          v[4 * q + 3] = w4.w;
        }
        tmem_st32(tmem + lane_off + X_COL + wg * 128 + j * 32, v);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->q_ready);
    }
    const uint32_t stg0 = sbase + OFF_STG + wg * HALF_BYTES;
    const bool issuer = (warp & 3) == 2;  // warp 2 / 6 copies its warpgroup's half
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    int n = 0;
    for (; n < N; ++n) {
      const int bb = n & 1;
      const int j0 = (t_lo + n) * T;
      if (!__all_sync(0xffffffffu, mbar_wait_cl(&bars->s_full[bb], (n >> 1) & 1, abort_flag, R))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld32(tmem + lane_off + S_COL + bb * T + cb0, *reinterpret_cast<uint32_t(*)[32]>(sr));
      tmem_ld32(tmem + lane_off + S_COL + bb * T + cb0 + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars->s_free[bb]);
      const bool full = (j0 >= band_key_lo(g, ihi)) && (j0 + T - 1 <= band_key_hi(g, i0));
      // visible key columns of row i in this tile, relative to this warpgroup's half
      const int clo = band_key_lo(g, i) - j0 - cb0;
      const int chi = band_key_hi(g, i) - j0 - cb0;
      const float pmax = full ? half_max<true>(sr, sl2, clo, chi) : half_max<false>(sr, sl2, clo, chi);
      xm[(bb * 2 + wg) * 128 + r] = pmax;
      mbar_arrive(&bars->mx[bb]);
      if (!__all_sync(0xffffffffu, mbar_wait_cl(&bars->mx[bb], (n >> 1) & 1, abort_flag, R))) {
        ok = false;
        break;
      }
      const float tmax = fmaxf(pmax, xm[(bb * 2 + (wg ^ 1)) * 128 + r]);
      float alpha = 1.f;
      if (tmax > m_run + kRescaleLog2) {
        if (m_run != -INFINITY) alpha = fast_exp2(m_run - tmax);
        m_run = tmax;
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      uint32_t pk[32];
      const float tsum = full ? half_p<true>(sr, sl2, m_use, clo, chi, pk) : half_p<false>(sr, sl2, m_use, clo, chi, pk);
      l_run = l_run * alpha + tsum;
      // the copy out of this staging half two steps ago (and of that alpha) must have landed
      if (n >= 2 &&
          !__all_sync(0xffffffffu, mbar_wait_cl(&bars->stg_free[bb][wg], ((n >> 1) - 1) & 1, abort_flag, R))) {
        ok = false;
        break;
      }
      const uint32_t stg = stg0 + bb * TILE_BYTES;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        st_smem_v4(stg + r * 128 + ((u ^ (r & 7)) << 4), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      if (wg == 0) alph[bb * 128 + r] = alpha;
      fence_proxy_async_smem();
      mbar_arrive(&bars->staged[wg]);
      if (issuer) {
        if (!__all_sync(0xffffffffu, mbar_wait_cl(&bars->staged[wg], n & 1, abort_flag, R) &&
                                         mbar_wait_cl(&bars->dst_free[bb], (n >> 1) & 1, abort_flag, R))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t full_bar = mapa(smem_u32(&bars->recv_full[bb]), 1);
          bulk_copy_to_cta(mapa(sbase + OFF_RECV + bb * TILE_BYTES + wg * HALF_BYTES, 1), stg, HALF_BYTES,
                           full_bar);
          if (wg == 0)
            bulk_copy_to_cta(mapa(sbase + OFF_RVEC + bb * 512, 1), smem_u32(alph + bb * 128), 512, full_bar);
          bars->n_sent[wg] = n + 1;
        }
      }
    }
    // row sum = the two warpgroups' partial sums (same running max); lse; send 1 / l
    xl[wg * 128 + r] = l_run;
    mbar_arrive(&bars->lx);
    if (ok && __all_sync(0xffffffffu, mbar_wait_cl(&bars->lx, 0, abort_flag, R))) {
      const float l_tot = xl[r] + xl[128 + r];
      if (wg == 0) {
        if (i < g.Lq) p.lse[(size_t)bh * g.Lq + i] = (m_run + log2f(l_tot)) * kLn2;
        finl[r] = 1.f / l_tot;
        fence_proxy_async_smem();
        mbar_arrive(&bars->fin_staged);
        if (issuer && __all_sync(0xffffffffu, mbar_wait_cl(&bars->fin_staged, 0, abort_flag, R)) && lane == 0) {
          bulk_copy_to_cta(mapa(sbase + OFF_RVEC + 1024, 1), smem_u32(finl), 512,
                           mapa(smem_u32(&bars->fin_full), 1));
          bars->fin_sent = 1;
        }
      }
    }
    // unwinding: the last copy out of the staging half must have been read
    if (!ok && issuer)
      for (int m = bars->n_sent[wg] - 1; m >= 0 && m >= bars->n_sent[wg] - 2; --m)
        mbar_wait_drain(&bars->stg_free[m & 1][wg], (m >> 1) & 1);
  } else {
    // ------------------------------------------------------------ rescale + epilogue (accumulator)
    const int wg = (warp - 2) >> 2, q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const int i = i0 + r;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const float* ralph = reinterpret_cast<const float*>(base + OFF_RVEC);  // [2][128]
    const float* rinv = ralph + 256;                                       // [128]
    bool ok = true;
    for (int n = 0; n < N; ++n) {
      const int bb = n & 1;
      if (!__all_sync(0xffffffffu, mbar_wait_cl(&bars->recv_full[bb], (n >> 1) & 1, abort_flag, R))) {
        ok = false;
        break;
      }
      if (threadIdx.x == 64) {
        bars->n_recv = n + 1;
        // both staging halves of the producer's tile n % 2 have been copied out
        mbar_arrive_remote(mapa(smem_u32(&bars->stg_free[bb][0]), 0));
        mbar_arrive_remote(mapa(smem_u32(&bars->stg_free[bb][1]), 0));
      }
      const float a = ralph[bb * 128 + r];
      if (__any_sync(0xffffffffu, a != 1.f)) {
        // O must hold PV of every earlier step before it is rescaled
        if (n >= 1 &&
            !__all_sync(0xffffffffu, mbar_wait_cl(&bars->mma_done[(n - 1) & 1], ((n - 1) >> 1) & 1, abort_flag, R))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {  // this warpgroup's 256 columns
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + 256 * wg + 32 * c, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * a);
          tmem_st32(tmem + lane_off + 256 * wg + 32 * c, v);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(&bars->o_ready[bb]);
    }
    if (ok && __all_sync(0xffffffffu, mbar_wait_cl(&bars->acc_done, 0, abort_flag, R) &&
                                         mbar_wait_cl(&bars->fin_full, 0, abort_flag, R))) {
      tc_fence_after();
      const float inv = rinv[r];
      const bool row_ok = i < g.Lq;
      float* orow = p.o + ((size_t)bh * g.Lq + (row_ok ? i : 0)) * DH;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        const int col = 256 * wg + 32 * c;
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + col, v);
        tmem_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(orow + col + e) =
                make_float4(__uint_as_float(v[e]) * inv, __uint_as_float(v[e + 1]) * inv,
                            __uint_as_float(v[e + 2]) * inv, __uint_as_float(v[e + 3]) * inv);
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA issues a copy or a remote arrival past this point
  if (!producer && threadIdx.x == 0) {
    // unwinding: tiles the producer sent that were never consumed must land
    // before this CTA's shared memory is released
    int sent0, sent1, fsent;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(sent0) : "r"(mapa(smem_u32(&bars->n_sent[0]), 0)) : "memory");
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(sent1) : "r"(mapa(smem_u32(&bars->n_sent[1]), 0)) : "memory");
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(fsent) : "r"(mapa(smem_u32(&bars->fin_sent), 0)) : "memory");
    const int sent = max(sent0, sent1);
    for (int m = bars->n_recv; m < sent; ++m) mbar_wait_drain(&bars->recv_full[m & 1], (m >> 1) & 1);
    if (fsent && *abort_flag) mbar_wait_drain(&bars->fin_full, 0);
  }
  __syncthreads();
  cluster_sync();
  if (*abort_flag && threadIdx.x == 0) atomicCAS(p.status, 0, kStatusTimeout);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_fwd_tc512_two_cta(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v16, float* o,
                             float* lse, int* status, cudaStream_t s) {
  CUtensorMap tk, tv;
  cudaError_t e;
  // 128-column slices of K and V: two 64-column chunks per TMA instruction
  if ((e = make_tmap_f16_chunks(&tk, k, DH, g.L, g.B * g.Hkv, T, 2)) != cudaSuccess) return e;
  if ((e = make_tmap_f16_chunks(&tv, v16, DH, g.L, g.B * g.Hkv, T, 2)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(fwd512_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM)) !=
      cudaSuccess)
    return e;
  FwdParams512 pm;
  pm.g = g;
  pm.q = q;
  pm.o = o;
  pm.lse = lse;
  pm.n_tiles = (g.Lq + T - 1) / T;
  pm.status = status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(R * (unsigned)g.G, (unsigned)pm.n_tiles, (unsigned)(g.B * g.Hkv));
  cfg.blockDim = dim3(kThr, 1, 1);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = R;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fwd512_kernel, tk, tv, pm);
}

}  // namespace swa
