// Tensor-core backward for head dim 512 on thread-block clusters.
//
// At D = 512 the two accumulators of a 128-key tile (dK and dV, 512 fp32
// columns each) need twice the Tensor Memory of one SM, and K plus V of the
// tile (128 KB each in fp16) do not fit one SM's shared memory together.  So
// the work of one tile is split by role across the CTAs of a cluster, each on
// its own SM:
//   producers (ranks 0 .. NP - 1, taking steps in turn): the resident A operand of
//     S lives in Tensor Memory (K for dK/dV, Q for dQ: 128 x 512 fp16 = 256
//     columns, read by TS-form MMAs), the resident A operand of dP in shared
//     memory (V, or dO); the streamed tiles come in 64-column slices.  They
//     form S and dP, then P = exp(scale S - lse) and dS = P (dP - Delta)
//     ("Training -- design (ORPO, flash-CCE head, prefix sharing, segmented
//     backward)", section 6: recompute P from the stored lse), and
//     bulk-copy the fp16 tiles into the accumulator CTAs' operand slots;
//   accumulators hold one full 128 x 512 fp32 accumulator in Tensor Memory:
//     dK/dV pass (NP + 2 CTAs per kv head and 128-row key tile, every query
//       head of the group and query tile in band):  rank NP  dV += P^T dO,
//       rank NP + 1  dK += dS^T Q;
//     dQ pass (NP + 1 CTAs per query head and query tile):  rank NP
//       dQ += dS K.
// Only tiles that meet the causal / window band are visited ("Lab 028 lab
// detail: Off NVIDIA, you fix the platform yourself", "What I changed, in
// plain terms" items 3-4).  A producer issues 2 x 2048 MMA cycles per own
// step and takes one step in NP; an accumulator issues 2048 per step.  A
// producer's own step takes about 11,000 cycles (shared-memory traffic of
// about 700 KB per own step, TMA issue and the copies), so three producers
// (NP = 3: 5-CTA dK/dV and 4-CTA dQ clusters) keep the accumulators busier
// than two, despite the SMs lost to cluster packing.  A producer moves one
// (dQ) or two (dK/dV) 32 KB tiles per own step over distributed shared
// memory (bulk copies).
//
// Warps: 0 TMA producer, 1 TMEM owner and MMA issuer, 2-9 elementwise (two
// warpgroups, 64 of the 128 columns each; a warpgroup stages its 64-column
// half of a tile and warp 2 / 6 issues the copy), 10 slot release
// (accumulator roles).  Every wait is bounded; a timeout in one CTA is
// broadcast to the whole cluster, every CTA drains its TMA loads, copies and
// MMAs in flight, and the status word records the timeout.
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

constexpr int kDirKV = 0, kDirQ = 1;
constexpr int kRoleProd = 0, kRoleAccP = 1, kRoleAccDS = 2;
constexpr int T = 128;     // tile rows on both sides (MMA M and N)
constexpr int DH = 512;    // head dim
constexpr int kThr = 352;  // 11 warps
constexpr int kSigWarp = 10;
constexpr float kLog2e = 1.4426950408889634f;

constexpr int RES_BYTES = T * DH * 2;  // resident dP A operand (V or dO), fp16
constexpr int TILE_BYTES = T * T * 2;  // fp16 128 x 128 operand tile
constexpr int HALF_BYTES = TILE_BYTES / 2;  // one warpgroup's 64-column half (one swizzle chunk)
constexpr int NR_P = 4;                // producer ring of 64-column slices
constexpr int SLOT_P = T * 64 * 2;
constexpr int SLOT_ACC = T * 128 * 2;  // accumulator ring of 128-column chunks
constexpr int OFF_STG = RES_BYTES;     // producer: two staging halves
constexpr int OFF_RING_P = RES_BYTES + 2 * HALF_BYTES;
constexpr int OFF_RECV = 0;            // accumulator: one operand slot per producer
constexpr int DATA_P = OFF_RING_P + NR_P * SLOT_P;
constexpr int kMaxNP = 3;
constexpr int kMaxRing = 5;
// accumulator layout for NP producers: NP operand slots, then as deep a ring
// as the producers' footprint allows
template <int NP>
struct AccLayout {
  static constexpr int OFF_RING = NP * TILE_BYTES;
  static constexpr int NR = (DATA_P - OFF_RING) / SLOT_ACC;
  static_assert(NR >= 2 && NR <= kMaxRing, "accumulator ring");
};
constexpr int DATA_BYTES = DATA_P;
static_assert(AccLayout<2>::OFF_RING + AccLayout<2>::NR * SLOT_ACC <= DATA_BYTES, "accumulator footprint");
static_assert(AccLayout<3>::OFF_RING + AccLayout<3>::NR * SLOT_ACC <= DATA_BYTES, "accumulator footprint");
// producer Tensor Memory: resident S operand, S, dP
constexpr uint32_t X_COL = 0, S_COL = 256, DP_COL = 384;

// A producer can be at most one step (of its own) ahead of an accumulator's
// release, so no cross-CTA barrier is ever more than one phase ahead of its
// waiter.
struct Bars {
  uint64_t res_full, x_ready;
  uint64_t ring_full[kMaxRing], ring_empty[kMaxRing];
  uint64_t t_full, t_free;      // (producer) S and dP in TMEM / read by the elementwise warps
  uint64_t staged[2];           // (producer) a warpgroup wrote its staging half
  uint64_t stg_free[2];         // (producer) the copy out of a staging half landed
  uint64_t dst_free[2];         // (producer) accumulator slot may be written: [0] P -> dV, [1] dS -> dK / dQ
  uint64_t recv_full[kMaxNP];   // (accumulator) tile from producer 0 .. NP - 1 landed
  uint64_t mma_done[kMaxNP];    // (accumulator) MMAs of a producer's step finished
  uint64_t acc_done, mma_drain;
  uint32_t tmem_slot;
  int abort_flag;
  int n_sent[2][2];             // (producer) steps copied to [dV, dK / dQ] by warpgroup [0, 1]
  int n_recv;                   // (accumulator) tiles received
};
static_assert(NR_P <= kMaxRing, "ring barriers");

constexpr size_t SMEM = (size_t)DATA_BYTES + 1024 + 1024;
static_assert(SMEM <= 232448, "shared memory");
static_assert(sizeof(Bars) <= 1024, "barrier block");

struct Params512 {
  Geom g;
  float* out0;             // KV: dk ; Q: dq
  float* out1;             // KV: dv
  const uint16_t* x16;     // resident S operand rows: KV: k16 ; Q: q16
  const float* stats;      // two planes: lse * log2e, then Delta (B * Hq * Lpad floats each)
  int Lpad;
  int n_tiles;
  int* status;
};

// P for 64 columns (cb0 .. cb0 + 63 of the tile) of one row, in place over the
// S values (fp32).  PER_COL: the lse belongs to the column (lse4 holds
// lse * log2e of the 64 columns, four per vector); otherwise l2 is the row's.
// Columns outside [clo, chi] are exactly zero unless FULL.
template <bool FULL, bool PER_COL>
__device__ __forceinline__ void p_tile64(uint32_t (&sv)[64], const float4* lse4, float l2, float sl2, int cb0,
                                         int clo, int chi) {
#pragma unroll
  for (int e = 0; e < 64; e += 4) {
    float lv[4] = {l2, l2, l2, l2};
    if (PER_COL) {
      const float4 l4 = __ldg(lse4 + (e >> 2));
      lv[0] = l4.x;
      lv[1] = l4.y;
      lv[2] = l4.z;
      lv[3] = l4.w;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float pv = fast_exp2(fmaf(__uint_as_float(sv[e + u]), sl2, -lv[u]));
      if (!FULL) pv = (cb0 + e + u >= clo && cb0 + e + u <= chi) ? pv : 0.f;
      sv[e + u] = __float_as_uint(pv);
    }
  }
}

__device__ __forceinline__ void pack64(const uint32_t (&v)[64], uint32_t (&o)[32]) {
#pragma unroll
  for (int e = 0; e < 64; e += 2) o[e >> 1] = pack_half2(__uint_as_float(v[e]), __uint_as_float(v[e + 1]));
}

// dS = P (dP - Delta) for 64 columns as fp16 pairs (dl4: Delta of the 64
// columns, four per vector, when PER_COL; otherwise dl is the row's).
template <bool PER_COL>
__device__ __forceinline__ void ds_tile64(const uint32_t (&pv)[64], const uint32_t (&dv)[64], const float4* dl4,
                                          float dl, uint32_t (&o)[32]) {
#pragma unroll
  for (int e = 0; e < 64; e += 4) {
    float dd[4] = {dl, dl, dl, dl};
    if (PER_COL) {
      const float4 d4 = __ldg(dl4 + (e >> 2));
      dd[0] = d4.x;
      dd[1] = d4.y;
      dd[2] = d4.z;
      dd[3] = d4.w;
    }
    o[e >> 1] = pack_half2(__uint_as_float(pv[e]) * (__uint_as_float(dv[e]) - dd[0]),
                           __uint_as_float(pv[e + 1]) * (__uint_as_float(dv[e + 1]) - dd[1]));
    o[(e >> 1) + 1] = pack_half2(__uint_as_float(pv[e + 2]) * (__uint_as_float(dv[e + 2]) - dd[2]),
                                 __uint_as_float(pv[e + 3]) * (__uint_as_float(dv[e + 3]) - dd[3]));
  }
}

template <int DIR, int NP>
__global__ void __launch_bounds__(kThr, 1)
    bwd512_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                  const Params512 p) {
  constexpr uint32_t R = NP + ((DIR == kDirKV) ? 2 : 1);  // CTAs per cluster
  constexpr int NR_ACC = AccLayout<NP>::NR;
  constexpr int OFF_RING_ACC = AccLayout<NP>::OFF_RING;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(base + DATA_BYTES);
  volatile int* abort_flag = &bars->abort_flag;
  const uint32_t sbase = smem_u32(base);

  const Geom& g = p.g;
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int role = rank < (uint32_t)NP ? kRoleProd : ((DIR == kDirKV && rank == (uint32_t)NP) ? kRoleAccP : kRoleAccDS);
  const bool acc_role = role != kRoleProd;
  // Grid (x, y, z) = (CTAs per cluster [x query heads of the group, dQ pass],
  // tiles, b * Hkv + kv head).  Blocks launch x fastest and z slowest, so the
  // clusters running at any moment share one kv head: its K and V (dQ pass)
  // or its group's Q and dO (dK/dV pass) are read from HBM about once and
  // then served by L2.
  const int bkv_z = (int)blockIdx.z;
  const int b = bkv_z / g.Hkv;
  const int head = (DIR == kDirKV) ? bkv_z  // b * Hkv + kv head
                                   : b * g.Hq + (bkv_z - b * g.Hkv) * g.G + (int)(blockIdx.x / R);  // query head
  // resident-side tile (keys for KV, queries for Q): longest band first
  const int tile = (DIR == kDirKV) ? (int)blockIdx.y : p.n_tiles - 1 - (int)blockIdx.y;
  const int r0 = tile * T;
  int t_lo, ntq, N;
  // rows of the resident side, and the last one that exists
  const int LX = (DIR == kDirKV) ? g.L : g.Lq;
  const int rlast = min(r0 + T, LX) - 1;
  if (DIR == kDirKV) {
    // query rows that can see a key of this tile
    const int qlo = band_q_lo(g, r0), qhi = band_q_hi(g, rlast);
    t_lo = qlo / T;
    ntq = qlo <= qhi ? qhi / T - t_lo + 1 : 0;
    N = g.G * ntq;
  } else {
    // key tiles meeting the band of rows r0 .. rlast (never empty)
    t_lo = band_key_lo(g, r0) / T;
    ntq = band_key_hi(g, rlast) / T - t_lo + 1;
    N = ntq;
  }
  if (N == 0) {
    // dK/dV pass, and no query sees these keys (queries that are a suffix of
    // the keys, with a window): zero gradients ("Lab 028 lab detail", "What
    // I changed, in plain terms" item 5(b)).  Every CTA of the cluster has
    // the same tile, so all of them leave here, before any cluster barrier.
    if (role == kRoleAccP) zero_rows(p.out1, head, r0, T, g.L, DH);
    if (role == kRoleAccDS) zero_rows(p.out0, head, r0, T, g.L, DH);
    return;
  }
  // streamed-side rows and head of step n.  dK/dV pass: query tiles from the
  // last one down, the group's query heads innermost, so that concurrent
  // clusters of one kv head (all starting at the last query tile) read the
  // same Q and dO tiles at about the same time.
  auto step_rows = [&](int n) {
    if (DIR == kDirKV) return (t_lo + ntq - 1 - n / g.G) * T;
    return (t_lo + n) * T;
  };
  auto step_head = [&](int n) -> int {
    if (DIR == kDirKV) return b * g.Hq + (head - b * g.Hkv) * g.G + n % g.G;  // query head
    return bkv_z;                                                              // kv head
  };
  // a producer takes steps n = rank, rank + NP, ...; m-th own step = rank + NP m
  const int n_own = role == kRoleProd ? max(0, (N - (int)rank + NP - 1) / NP) : 0;
  // accumulator: which of the producer's two destinations this CTA is
  const int dst_kind = (role == kRoleAccP) ? 0 : 1;

  if (threadIdx.x == 0) {
    mbar_init(&bars->res_full, 1);
    mbar_init(&bars->x_ready, 256);
    for (int s = 0; s < kMaxRing; ++s) {
      mbar_init(&bars->ring_full[s], 1);
      mbar_init(&bars->ring_empty[s], 1);
    }
    mbar_init(&bars->t_full, 1);
    mbar_init(&bars->t_free, 256);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->staged[s], 128);
      mbar_init(&bars->stg_free[s], 1);
      mbar_init(&bars->dst_free[s], 1);
      bars->n_sent[s][0] = bars->n_sent[s][1] = 0;
    }
    for (int s = 0; s < kMaxNP; ++s) {
      mbar_init(&bars->recv_full[s], 1);
      mbar_init(&bars->mma_done[s], 1);
    }
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->mma_drain, 1);
    bars->abort_flag = 0;
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
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmG);
      int issued = 0;  // ring loads issued
      bool ok = true;
      if (!acc_role) {
        // resident dP operand, then per own step 8 slices for S and 8 for dP
        const CUtensorMap* mres = (DIR == kDirKV) ? &tmV : &tmG;
        const CUtensorMap* ms = (DIR == kDirKV) ? &tmQ : &tmK;
        const CUtensorMap* mp = (DIR == kDirKV) ? &tmG : &tmV;
        mbar_arrive_expect_tx(&bars->res_full, RES_BYTES);
        for (int c = 0; c < DH / 64; ++c) tma_load_3d(base + c * T * 128, mres, &bars->res_full, c * 64, r0, head);
        for (int m = 0; ok && m < n_own; ++m) {
          const int n = (int)rank + NP * m;
          const int rows = step_rows(n), hd = step_head(n);
          for (int k = 0; k < 2 * (DH / 64); ++k, ++issued) {
            const int s = issued % NR_P;
            if (issued >= NR_P && !mbar_wait_cl(&bars->ring_empty[s], ((issued / NR_P) & 1) ^ 1, abort_flag, R)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&bars->ring_full[s], SLOT_P);
            tma_load_3d(base + OFF_RING_P + s * SLOT_P, (k & 1) ? mp : ms, &bars->ring_full[s], (k >> 1) * 64, rows,
                        hd);
          }
        }
        if (!ok) mbar_wait_drain(&bars->res_full, 0);
      } else {
        // 128-column chunks of dO (dV), Q (dK) or K (dQ)
        const CUtensorMap* mstr = (role == kRoleAccP) ? &tmG : ((DIR == kDirKV) ? &tmQ : &tmK);
        for (int n = 0; ok && n < N; ++n) {
          const int rows = step_rows(n), hd = step_head(n);
          for (int c = 0; c < DH / 128; ++c, ++issued) {
            const int s = issued % NR_ACC;
            if (issued >= NR_ACC &&
                !mbar_wait_cl(&bars->ring_empty[s], ((issued / NR_ACC) & 1) ^ 1, abort_flag, R)) {
              ok = false;
              break;
            }
            unsigned char* dst = base + OFF_RING_ACC + s * SLOT_ACC;
            mbar_arrive_expect_tx(&bars->ring_full[s], SLOT_ACC);
            tma_load_3d(dst, mstr, &bars->ring_full[s], c * 128, rows, hd);
            tma_load_3d(dst + T * 128, mstr, &bars->ring_full[s], c * 128 + 64, rows, hd);
          }
        }
      }
      if (!ok) {
        // unwinding: let the loads in flight land (at most one per slot)
        const int nr = acc_role ? NR_ACC : NR_P;
        for (int k = issued - 1; k >= 0 && k >= issued - nr; --k)
          mbar_wait_drain(&bars->ring_full[k % nr], (k / nr) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      bool ok = true;
      const uint32_t idS = idesc_f16(T, T, 0, 0, 0, 0);  // both operands K-major
      if (!acc_role) {
        const uint64_t yd = smem_desc_sw128(sbase, 16, 1024);  // resident dP operand
        ok = mbar_wait_cl(&bars->res_full, 0, abort_flag, R) && mbar_wait_cl(&bars->x_ready, 0, abort_flag, R);
        int used = 0;
        for (int m = 0; ok && m < n_own; ++m) {
          if (m >= 1 && !mbar_wait_cl(&bars->t_free, (m - 1) & 1, abort_flag, R)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int k = 0; k < 2 * (DH / 64); ++k, ++used) {
            const int s = used % NR_P, c = k >> 1;
            if (!mbar_wait_cl(&bars->ring_full[s], (used / NR_P) & 1, abort_flag, R)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t sd = smem_desc_sw128(sbase + OFF_RING_P + s * SLOT_P, 16, 1024);
            if ((k & 1) == 0) {
              // S += X[:, 64c .. 64c + 63] slice^T, X from Tensor Memory (8 columns per 16 elements)
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                mma_ts(tmem + S_COL, tmem + X_COL + c * 32 + ks * 8, desc_add(sd, ks * 32), idS, (c | ks) ? 1u : 0u);
            } else {
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                mma_ss(tmem + DP_COL, desc_add(yd, c * T * 128 + ks * 32), desc_add(sd, ks * 32), idS,
                       (c | ks) ? 1u : 0u);
            }
            mma_commit(&bars->ring_empty[s]);
          }
          if (!ok) break;
          mma_commit(&bars->t_full);
        }
      } else {
        const uint32_t idA = idesc_f16(T, 128, 0, 0, 0, 1);  // A K-major (fp16 tile), B MN-major
        int used = 0;
        for (int n = 0; ok && n < N; ++n) {
          const int s2 = n % NP;  // producer of step n, and its slot
          if (!mbar_wait_cl(&bars->recv_full[s2], (n / NP) & 1, abort_flag, R)) {
            ok = false;
            break;
          }
          bars->n_recv = n + 1;
          tc_fence_after();
          const uint64_t ad = smem_desc_sw128(sbase + OFF_RECV + s2 * TILE_BYTES, 16, 1024);
          for (int c = 0; c < DH / 128; ++c, ++used) {
            const int s = used % NR_ACC;
            if (!mbar_wait_cl(&bars->ring_full[s], (used / NR_ACC) & 1, abort_flag, R)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t bd = smem_desc_sw128(sbase + OFF_RING_ACC + s * SLOT_ACC, T * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < T / 16; ++ks)
              mma_ss(tmem + c * 128, desc_add(ad, (ks >> 2) * T * 128 + (ks & 3) * 32), desc_add(bd, ks * 2048),
                     idA, (n | ks) ? 1u : 0u);
            mma_commit(&bars->ring_empty[s]);
          }
          if (!ok) break;
          mma_commit(&bars->mma_done[s2]);
        }
        if (ok) mma_commit(&bars->acc_done);
      }
      // every MMA issued so far has finished before TMEM is released
      mma_commit(&bars->mma_drain);
      mbar_wait_drain(&bars->mma_drain, 0);
    }
  } else if (warp == kSigWarp) {
    // ------------------------------------------------------------ slot release (accumulator roles)
    if (acc_role && elect_one()) {
      // arm each producer's slot for its first step, then re-arm after each step's MMAs
      for (int s = 0; s < NP && s < N; ++s) {
        mbar_arrive_expect_tx(&bars->recv_full[s], TILE_BYTES);
        mbar_arrive_remote(mapa(smem_u32(&bars->dst_free[dst_kind]), (uint32_t)s));
      }
      for (int n = 0; n + NP < N; ++n) {
        const int s2 = n % NP;
        if (!mbar_wait_cl(&bars->mma_done[s2], (n / NP) & 1, abort_flag, R)) break;
        mbar_arrive_expect_tx(&bars->recv_full[s2], TILE_BYTES);
        mbar_arrive_remote(mapa(smem_u32(&bars->dst_free[dst_kind]), (uint32_t)s2));
      }
    }
  } else if (!acc_role) {
    // ------------------------------------------------------------ elementwise (producers)
    const int wg = (warp - 2) >> 2, q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const float sl2 = g.scale * kLog2e;
    const int cb0 = 64 * wg;
    const int row = r0 + r;  // key (KV) or query (Q) of this thread
    {
      // resident S operand into Tensor Memory: row r, fp16 pairs -> one 32-bit column each;
      // warpgroup wg fills columns [128 wg, 128 wg + 128) (head-dim elements [256 wg, 256 wg + 256))
      const uint4* src = reinterpret_cast<const uint4*>(p.x16 + ((size_t)head * LX + (row < LX ? row : 0)) * DH) +
                         wg * 32;
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        uint32_t v[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 w4 = row < LX ? __ldg(src + j * 8 + q) : make_uint4(0u, 0u, 0u, 0u);
          v[4 * q] = w4.x;
          v[4 * q + 1] = w4.y;
          v[4 * q + 2] = w4.z;
          v[4 * q + 3] = w4.w;
        }
        tmem_st32(tmem + lane_off + X_COL + wg * 128 + j * 32, v);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->x_ready);
    }
    float2 rs_row = make_float2(0.f, 0.f);
    if (DIR == kDirQ)
      rs_row = make_float2(p.stats[(size_t)head * p.Lpad + row], p.stats[((size_t)g.B * g.Hq + head) * p.Lpad + row]);
    const uint32_t stg = sbase + OFF_STG + wg * HALF_BYTES;
    const uint32_t stg_row = stg + r * 128;
    const bool issuer = (warp & 3) == 2;  // warp 2 / 6 copies its warpgroup's half
    int copies = 0;                       // copies out of this warpgroup's staging half
    bool ok = true;
    // stage one 64-column half tile and copy it into accumulator rank `dst`'s slot
    auto send = [&](const uint32_t (&o)[32], int kind, uint32_t dst, int m) -> bool {
      if (copies > 0 && !__all_sync(0xffffffffu, mbar_wait_cl(&bars->stg_free[wg], (copies - 1) & 1, abort_flag, R)))
        return false;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        st_smem_v4(stg_row + ((u ^ (r & 7)) << 4), o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
      fence_proxy_async_smem();
      mbar_arrive(&bars->staged[wg]);
      if (issuer) {
        if (!__all_sync(0xffffffffu, mbar_wait_cl(&bars->staged[wg], copies & 1, abort_flag, R) &&
                                         mbar_wait_cl(&bars->dst_free[kind], m & 1, abort_flag, R)))
          return false;
        if (lane == 0) {
          bulk_copy_to_cta(mapa(sbase + OFF_RECV + rank * TILE_BYTES + wg * HALF_BYTES, dst), stg, HALF_BYTES,
                           mapa(smem_u32(&bars->recv_full[rank]), dst));
          bars->n_sent[kind][wg] = m + 1;
        }
      }
      ++copies;
      return true;
    };
    for (int m = 0; m < n_own; ++m) {
      const int n = (int)rank + NP * m;
      const int c0 = step_rows(n);  // first column's query (KV) or key (Q)
      const float4 *lse4 = nullptr, *dl4 = nullptr;
      if (DIR == kDirKV) {
        const float* lse_g = p.stats + (size_t)step_head(n) * p.Lpad + c0 + cb0;
        lse4 = reinterpret_cast<const float4*>(lse_g);
        dl4 = reinterpret_cast<const float4*>(lse_g + (size_t)g.B * g.Hq * p.Lpad);
      }
      if (!__all_sync(0xffffffffu, mbar_wait_cl(&bars->t_full, m & 1, abort_flag, R))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[64], dv[64];
      tmem_ld32(tmem + lane_off + S_COL + cb0, *reinterpret_cast<uint32_t(*)[32]>(sv));
      tmem_ld32(tmem + lane_off + S_COL + cb0 + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
      tmem_ld32(tmem + lane_off + DP_COL + cb0, *reinterpret_cast<uint32_t(*)[32]>(dv));
      tmem_ld32(tmem + lane_off + DP_COL + cb0 + 32, *reinterpret_cast<uint32_t(*)[32]>(dv + 32));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars->t_free);  // S and dP may be overwritten by the next own step
      bool full;
      int clo, chi;
      if (DIR == kDirKV) {  // columns are query rows c0 .. c0 + 127, this thread's row is key `row`
        full = (c0 >= band_q_lo(g, rlast)) && (c0 + T - 1 <= band_q_hi(g, r0));
        clo = band_q_lo(g, row) - c0;
        chi = band_q_hi(g, row) - c0;
      } else {  // columns are keys c0 .. c0 + 127, this thread's row is query `row`
        full = (c0 >= band_key_lo(g, rlast)) && (c0 + T - 1 <= band_key_hi(g, r0));
        clo = band_key_lo(g, row) - c0;
        chi = band_key_hi(g, row) - c0;
      }
      if (full) p_tile64<true, DIR == kDirKV>(sv, lse4, rs_row.x, sl2, cb0, clo, chi);
      else p_tile64<false, DIR == kDirKV>(sv, lse4, rs_row.x, sl2, cb0, clo, chi);
      uint32_t o[32];
      if (DIR == kDirKV) {
        pack64(sv, o);
        if (!send(o, 0, (uint32_t)NP, m)) {  // P^T -> dV accumulator
          ok = false;
          break;
        }
      }
      ds_tile64<DIR == kDirKV>(sv, dv, dl4, rs_row.y, o);
      if (!send(o, 1, DIR == kDirKV ? (uint32_t)NP + 1 : (uint32_t)NP, m)) {  // dS -> dK / dQ accumulator
        ok = false;
        break;
      }
    }
    // unwinding: the last copy out of the staging half must have been read
    if (!ok && issuer && copies > 0) mbar_wait_drain(&bars->stg_free[wg], (copies - 1) & 1);
  } else {
    // ------------------------------------------------------------ epilogue (accumulator roles)
    const int wg = (warp - 2) >> 2, q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    if (warp == 2 && elect_one()) {
      // as soon as a producer's tile has landed, both of its staging halves may
      // be rewritten: tell it then, not when the MMA thread reaches the step
      for (int n = 0; n < N; ++n) {
        const int s2 = n % NP;
        if (!mbar_wait_cl(&bars->recv_full[s2], (n / NP) & 1, abort_flag, R)) break;
        mbar_arrive_remote(mapa(smem_u32(&bars->stg_free[0]), (uint32_t)s2));
        mbar_arrive_remote(mapa(smem_u32(&bars->stg_free[1]), (uint32_t)s2));
      }
    }
    __syncwarp();
    if (__all_sync(0xffffffffu, mbar_wait_cl(&bars->acc_done, 0, abort_flag, R))) {
      tc_fence_after();
      const int row = r0 + r;
      const bool row_ok = row < LX;
      float* dst;
      float mul;
      if (DIR == kDirKV) {
        dst = (role == kRoleAccP) ? p.out1 : p.out0;
        mul = (role == kRoleAccP) ? 1.f : g.scale;
      } else {
        dst = p.out0;
        mul = g.scale;
      }
      dst += ((size_t)head * LX + (row_ok ? row : 0)) * DH;
#pragma unroll 1
      for (int cc = 0; cc < 8; ++cc) {
        const int c = 256 * wg + 32 * cc;
        uint32_t a[32];
        tmem_ld32(tmem + lane_off + c, a);
        tmem_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(dst + c + e) =
                make_float4(__uint_as_float(a[e]) * mul, __uint_as_float(a[e + 1]) * mul,
                            __uint_as_float(a[e + 2]) * mul, __uint_as_float(a[e + 3]) * mul);
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA issues a copy or a remote arrival past this point
  if (acc_role && threadIdx.x == 0) {
    // unwinding: tiles the producers sent that were never consumed must land
    // before this CTA's shared memory is released
    for (uint32_t pr = 0; pr < (uint32_t)NP; ++pr) {
      int sent0, sent1;
      asm volatile("ld.shared::cluster.u32 %0, [%1];"
                   : "=r"(sent0)
                   : "r"(mapa(smem_u32(&bars->n_sent[dst_kind][0]), pr))
                   : "memory");
      asm volatile("ld.shared::cluster.u32 %0, [%1];"
                   : "=r"(sent1)
                   : "r"(mapa(smem_u32(&bars->n_sent[dst_kind][1]), pr))
                   : "memory");
      const int sent = max(sent0, sent1);  // a step with either half in flight
      // producer pr sent its own steps 0 .. sent - 1, i.e. steps pr + NP m
      for (int m = 0; m < sent; ++m) {
        const int n = (int)pr + NP * m;
        if (n >= bars->n_recv) mbar_wait_drain(&bars->recv_full[pr], m & 1);
      }
    }
  }
  __syncthreads();
  cluster_sync();
  if (*abort_flag && threadIdx.x == 0) atomicCAS(p.status, 0, kStatusTimeout);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DIR, int NP>
cudaError_t launch_dir(const Geom& g, const uint16_t* q16, const uint16_t* k16, const uint16_t* v16,
                       const uint16_t* g16, const float* stats, int Lpad, float* out0, float* out1, int* status,
                       cudaStream_t s) {
  CUtensorMap tq, tk, tv, tg;
  cudaError_t e;
  if ((e = make_tmap_f16(&tq, q16, DH, g.Lq, g.B * g.Hq, T)) != cudaSuccess) return e;
  if ((e = make_tmap_f16(&tg, g16, DH, g.Lq, g.B * g.Hq, T)) != cudaSuccess) return e;
  if ((e = make_tmap_f16(&tk, k16, DH, g.L, g.B * g.Hkv, T)) != cudaSuccess) return e;
  if ((e = make_tmap_f16(&tv, v16, DH, g.L, g.B * g.Hkv, T)) != cudaSuccess) return e;
  auto kern = bwd512_kernel<DIR, NP>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM)) != cudaSuccess)
    return e;
  Params512 pm;
  pm.g = g;
  pm.out0 = out0;
  pm.out1 = out1;
  pm.x16 = (DIR == kDirKV) ? k16 : q16;
  pm.stats = stats;
  pm.Lpad = Lpad;
  pm.n_tiles = ((DIR == kDirKV ? g.L : g.Lq) + T - 1) / T;  // resident-side tiles
  pm.status = status;
  const unsigned R = NP + ((DIR == kDirKV) ? 2 : 1);
  const unsigned xs = (DIR == kDirKV) ? R : R * (unsigned)g.G;  // dQ pass: the group's query heads along x
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(xs, (unsigned)pm.n_tiles, (unsigned)(g.B * g.Hkv));
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
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, tg, pm);
}

}  // namespace

cudaError_t launch_bwd_dkdv_tc512(const Geom& g, const uint16_t* q16, const uint16_t* k16, const uint16_t* v16,
                                  const uint16_t* g16, const float* stats, int Lpad, float* dk, float* dv,
                                  int* status, cudaStream_t s) {
  return launch_dir<kDirKV, 3>(g, q16, k16, v16, g16, stats, Lpad, dk, dv, status, s);
}

cudaError_t launch_bwd_dq_tc512(const Geom& g, const uint16_t* q16, const uint16_t* k16, const uint16_t* v16,
                                const uint16_t* g16, const float* stats, int Lpad, float* dq, int* status,
                                cudaStream_t s) {
  return launch_dir<kDirQ, 3>(g, q16, k16, v16, g16, stats, Lpad, dq, nullptr, status, s);
}

}  // namespace swa
