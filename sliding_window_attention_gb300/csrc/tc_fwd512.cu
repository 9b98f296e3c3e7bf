// Tensor-core forward for head dim 512 on clusters of CTA pairs.
//
// At D = 512 the output accumulator O of a 128-row query tile (512 fp32
// columns) fills one SM's Tensor Memory, so S and O cannot live on the same
// SM.  Persistent 4-CTA clusters, as many as fit on the GPU, loop over work
// items of (query head, two adjacent 128-row query tiles), longest rows first
// (cluster_items.cuh); the next item's Q is loaded while the accumulator
// writes the previous item's O.  Every role runs on a CTA pair (tcgen05 .cta_group::2):
// each CTA of a pair owns one of the two query tiles, and each MMA of M = 256
// rows takes its B operand half from each CTA, so every K and V tile crosses
// each SM's TMA engine and shared memory once per pair, half in each CTA.
//   producers (ranks 0-1): Q sits in Tensor Memory as fp16 pairs (256
//     columns, the A operand of TS-form MMAs); each CTA streams its 64-key
//     half of the step's K tile in 32 KB slices of 256 columns; S = Q K^T
//     (N = 128 keys) into two TMEM buffers; online softmax with the band mask
//     on edge tiles ("Lab 028 lab detail: Off NVIDIA, you fix the platform
//     yourself", "What I changed, in plain terms" items 3-4); P in fp16 is
//     staged (two staging tiles, so a tile is stored while the next P is
//     formed) and handed, with the per-row factor by which O must be
//     rescaled, to the accumulator CTA of the same half through an L2 scratch
//     (below); at the end each CTA writes its rows' logsumexp (same section,
//     item 1) and sends 1 / l.
//   accumulators (ranks 2-3): O (512 columns) in Tensor Memory; each CTA
//     streams its 128-column half of each 256-column V chunk; before O += P V
//     of a step its elementwise warps rescale the rows whose running maximum
//     moved (the maximum moves lazily, only when it grows by more than 2^8,
//     so this is rare); at the end it writes O / l.
// The pair's even CTA (the leader) issues the pair's MMAs; the peer's warps
// arrive locally and one relay warp forwards one arrival per step.
//
// Warps: 0 TMA, 1 TMEM owner and (leader) MMA issuer, 2-9 elementwise (two
// warpgroups, 64 columns of S or 256 columns of O each), 10 tile loads
// (accumulators), relay (producer peer) or the work-item scheduler (rank 0),
// 11 tile stores (producers) or relay (accumulator peer).  Every wait is bounded; a timeout in one CTA is
// broadcast to the cluster, every CTA drains its loads, stores, copies and
// MMAs, and the status word records it.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "swa_internal.h"
#include "cluster_items.cuh"
#include "tc_ptx.cuh"

namespace swa {
namespace {

using namespace tc;

constexpr int T = 128;     // query rows per tile and keys per step
constexpr int HT = 64;     // keys per CTA per step (producers)
constexpr int DH = 512;    // head dim
constexpr int kThr = 384;  // 12 warps
constexpr int kSigWarp = 10, kRelayWarp = 11;  // 11: tile stores in producers, relay in accumulators
constexpr uint32_t R = 4;  // CTAs per cluster
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kMaxDevices = 64;

constexpr int TILE_BYTES = T * T * 2;       // fp16 128 x 128 P tile
constexpr int HALF_BYTES = TILE_BYTES / 2;  // one warpgroup's 64 columns (one swizzle chunk)
// producer shared memory: two staging tiles, row vectors, K ring of 32 KB
// slices (four 64-column chunks of this CTA's 64 keys)
constexpr int OFF_STG = 0;
constexpr int OFF_VEC = 2 * TILE_BYTES;  // alpha[2][128], (free)[128], max exchange [2][2][128], l exchange [2][128], 1 / l [2][128]
constexpr int OFF_RING_P = OFF_VEC + 8192;
constexpr int SLOT_P = HT * 256 * 2;
constexpr int NR_P = 4;
// accumulator shared memory: two P slots, two alpha slots + 1 / l, V ring of
// 32 KB slots (two 64-column chunks of the 128 keys)
constexpr int OFF_RECV = 0;
constexpr int OFF_RVEC = 2 * TILE_BYTES;  // alpha slot [2][128], inv_l [2 item parity][128]
constexpr int OFF_RING_A = 2 * TILE_BYTES + 2048;
constexpr int SLOT_A = T * 128 * 2;
constexpr int NR_A = 4;
constexpr int DATA_P = OFF_RING_P + NR_P * SLOT_P;
constexpr int DATA_A = OFF_RING_A + NR_A * SLOT_A;
constexpr int DATA_BYTES = DATA_P > DATA_A ? DATA_P : DATA_A;
constexpr int kMaxRing = NR_P > NR_A ? NR_P : NR_A;
constexpr uint32_t X_COL = 0, S_COL = 256;  // producer TMEM: Q [0, 256), S buffers [256, 512)
static_assert(OFF_VEC + 1024 + 512 + 2048 + 1024 + 1024 <= OFF_RING_P, "producer vectors");

// Producer -> accumulator P tiles (with their row factors) travel through L2:
// a producer warp bulk-stores the staged tile into the scratch of the
// accumulator CTA's SM (the staging is free as soon as the store has read
// it) and the accumulator bulk-loads it into its operand slot.  One CTA of
// this kernel fills an SM, so the scratch of an SM belongs to one
// accumulator CTA at a time: two slots of a 32 KB tile + 512 B of factors.
constexpr int kScratchSms = 192;
constexpr int SCR_SLOT = TILE_BYTES + 1024;
__device__ __align__(1024) unsigned char g_fwd_tile_scratch[(size_t)kScratchSms * 2 * SCR_SLOT];
static_assert(OFF_RING_A % 1024 == 0 && OFF_RING_P % 1024 == 0, "swizzled tiles need 1 KB alignment");

struct Bars {
  uint64_t ring_full[kMaxRing];  // (leader) both halves of a slot landed
  uint64_t ring_empty[kMaxRing]; // (both) the pair's MMAs finished reading a slot
  uint64_t q_ready;              // (producer, own) an item's Q in TMEM
  uint64_t pair_ready;           // (producer leader) both CTAs' Q in TMEM
  uint64_t s_full[2], s_free[2]; // (producer) S buffers: filled (both) / read (leader: 8 warps + relay)
  uint64_t mx[2][4];             // (producer) both warps of lane quarter q posted their partial row max [parity][q]
  uint64_t staged[2][2];         // (producer) a warpgroup's 4 warps wrote its half of staging tile [tile][warpgroup]
  uint64_t stg_free[2][2];       // (producer) the store warp has read staging half [tile][warpgroup] out
  uint64_t scratch_free[2];      // (producer) the accumulator loaded scratch slot
  uint64_t tile_ready[2];        // (accumulator) the producer's tile for slot is in the scratch
  uint64_t recv_full[2];         // (accumulator) P tile + alpha landed in slot
  uint64_t o_ready[2];           // (accumulator) rows rescaled for the step (leader: 8 warps + relay)
  uint64_t mma_done[2];          // (accumulator, both) PV of a slot finished
  uint64_t lx;                   // (producer) both warpgroups posted an item's row sums
  uint64_t fin_staged;           // (producer) an item's 1 / l written
  uint64_t fin_full[2];          // (accumulator) an item's 1 / l landed [item parity]
  uint64_t acc_done;             // (accumulator, both) an item's PV MMAs finished
  uint64_t acc_free;             // (accumulator leader) both CTAs read an item's O out
  uint64_t epi_done;             // (accumulator, own) the epilogue's stores read their staging
  uint64_t mma_drain;
  uint32_t tmem_slot;
  int abort_flag;
  int n_sent[2];                 // (producer) steps copied, per warpgroup
  int fin_sent;                  // (producer) 1 / l copies issued
  int n_recv;                    // (accumulator) steps whose tile landed
  int n_loaded;                  // (accumulator) steps whose tile loads were issued
  int smid;                      // (accumulator) SM this CTA runs on: the scratch it loads from
  int n_issued;                  // ring loads issued by this CTA
  ItemRing items;                // work-item ids from rank 0's scheduler
};

constexpr size_t SMEM = (size_t)DATA_BYTES + 1024 + 1024;
static_assert(SMEM <= 232448, "shared memory");
static_assert(sizeof(Bars) <= 1024, "barrier block");

struct FwdPairParams {
  Geom g;
  int* work;          // the launch's work counter: the next item id (zero before the launch)
  int n_items;        // work items
  const uint16_t* q;  // bf16: S = Q K^T reads the caller's q and k as they are
  float* o;
  float* lse;
  int n_tiles;        // 128-row query tiles
  int* status;
};

// Scaled maximum over 64 raw scores of one row; entries outside the row's
// visible columns v (see vis(); TWO under a shared-prefix plan) are excluded
// unless FULL (correct for any sign of the scale).
template <bool FULL, bool TWO = false>
__device__ __forceinline__ float half_max(const uint32_t (&sr)[64], float sl2, const int4& v) {
  float a0 = -INFINITY, a1 = -INFINITY;
#pragma unroll
  for (int e = 0; e < 64; e += 2) {
    float x0 = __uint_as_float(sr[e]) * sl2, x1 = __uint_as_float(sr[e + 1]) * sl2;
    if (!FULL) {
      x0 = vis<TWO>(e, v) ? x0 : -INFINITY;
      x1 = vis<TWO>(e + 1, v) ? x1 : -INFINITY;
    }
    a0 = fmaxf(a0, x0);
    a1 = fmaxf(a1, x1);
  }
  return fmaxf(a0, a1);
}

// Maximum over 64 raw scores of one row, same exclusions as half_max.  For a
// positive scale, half_max_raw * sl2 equals half_max exactly (rounding is
// monotonic); three-input max halves the instructions.
template <bool FULL, bool TWO = false>
__device__ __forceinline__ float half_max_raw(const uint32_t (&sr)[64], const int4& v) {
  float a0 = -INFINITY, a1 = -INFINITY;
#pragma unroll
  for (int e = 0; e < 64; e += 4) {
    float x[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[k] = __uint_as_float(sr[e + k]);
      if (!FULL) x[k] = vis<TWO>(e + k, v) ? x[k] : -INFINITY;
    }
    a0 = fmax3(a0, x[0], x[1]);
    a1 = fmax3(a1, x[2], x[3]);
  }
  return fmaxf(a0, a1);
}

// P = 2^(sl2 s - m) for 64 entries as fp16 pairs; returns the fp32 row sum.
// The scaling and the two running sums (even and odd entries) use paired
// .f32x2 instructions: same roundings as scalar fmaf / adds, half the issue
// slots.
template <bool FULL, bool TWO = false>
__device__ __forceinline__ float half_p(const uint32_t (&sr)[64], float sl2, float m_use, const int4& v,
                                        uint32_t (&pk)[32]) {
  const uint64_t sc = f2_pack(sl2, sl2), nm = f2_pack(-m_use, -m_use);
  uint64_t acc = f2_pack(0.f, 0.f);
#pragma unroll
  for (int e = 0; e < 64; e += 2) {
    const float2 x = f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sc, nm));
    float p0 = fast_exp2(x.x);
    float p1 = fast_exp2(x.y);
    if (!FULL) {
      p0 = vis<TWO>(e, v) ? p0 : 0.f;
      p1 = vis<TWO>(e + 1, v) ? p1 : 0.f;
    }
    acc = f2_add(acc, f2_pack(p0, p1));
    pk[e >> 1] = pack_half2(p0, p1);
  }
  const float2 t = f2_unpack(acc);
  return t.x + t.y;
}

// One work item of a persistent cluster: two adjacent 128-row query tiles of
// one query head.  Ids run with the kv head (b * Hkv + kv head) slowest, then
// the tile pair (the longest band first), then the group's query head, so
// that the clusters working at any moment share one kv head, whose K and V
// then stay in L2, and the short items come last.
struct FwdItem {
  int bkv, bh;      // b * Hkv + kv head; b * Hq + query head
  int i0, ihi;      // this CTA's query tile (ihi = i0 when it has no rows)
  bool own_rows;    // false for the second tile of an odd last pair
  TileSteps ks;     // key tiles meeting the band of the pair's rows (at least one)
  int N;
};

__device__ __forceinline__ FwdItem make_fwd_item(const Geom& g, int id, int npairs, uint32_t h) {
  FwdItem x;
  const int per_kv = npairs * g.G;
  x.bkv = id / per_kv;
  const int rem = id - x.bkv * per_kv;
  const int y = rem / g.G;
  const int b = x.bkv / g.Hkv;
  x.bh = b * g.Hq + (x.bkv - b * g.Hkv) * g.G + (rem - y * g.G);
  const int tp = npairs - 1 - y;  // the last query tile pair has the longest band
  const int pr0 = 2 * tp * T, prlast = min(pr0 + 2 * T, g.Lq) - 1;
  x.i0 = pr0 + (int)h * T;
  x.own_rows = x.i0 < g.Lq;
  x.ihi = x.own_rows ? min(x.i0 + T, g.Lq) - 1 : x.i0;
  x.ks = row_steps(g, pr0, prlast, T);
  x.N = x.ks.count();
  return x;
}

// Readers of each item id in a cluster (the scheduler counts their arrivals
// before it reuses the id's slot): the producer leader's TMA, MMA, eight
// elementwise and store warps (11), the producer peer's same plus its relay
// warp (12), the accumulator leader's TMA, MMA, tile-load and eight
// elementwise warps (11), the accumulator peer's TMA, tile-load, eight
// elementwise and relay warps (11).
constexpr int kItemReaders = 11 + 12 + 11 + 11;

__global__ void __launch_bounds__(kThr, 1)
    fwd512_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmO,  // fp32 o, 32 x 32 boxes
                   const FwdPairParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(base + DATA_BYTES);
  volatile int* abort_flag = &bars->abort_flag;
  const uint32_t sbase = smem_u32(base);

  const Geom& g = p.g;
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const uint32_t h = rank & 1u;      // half of the pair: which query tile, which keys / columns
  const uint32_t lead = rank & ~1u;  // the pair's leader
  const bool leader = h == 0;
  const uint16_t pmask = (uint16_t)(3u << lead);
  const bool producer = rank < 2;
  const int npairs = (p.n_tiles + 1) / 2;
  const bool two = g.Rc > 0;  // shared-prefix plan: two visible key intervals per row

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxRing; ++s) {
      mbar_init(&bars->ring_full[s], 1);
      mbar_init(&bars->ring_empty[s], 1);
    }
    mbar_init(&bars->q_ready, 256);
    mbar_init(&bars->pair_ready, 2);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->s_free[s], leader ? 9 : 8);
      for (int q = 0; q < 4; ++q) mbar_init(&bars->mx[s][q], 2);  // one arrival per warp
      mbar_init(&bars->staged[s][0], 4);
      mbar_init(&bars->staged[s][1], 4);
      mbar_init(&bars->stg_free[s][0], 1);
      mbar_init(&bars->stg_free[s][1], 1);
      mbar_init(&bars->scratch_free[s], 1);
      mbar_init(&bars->tile_ready[s], 1);
      mbar_init(&bars->recv_full[s], 1);
      mbar_init(&bars->o_ready[s], leader ? 9 : 8);
      mbar_init(&bars->mma_done[s], 1);
      mbar_init(&bars->fin_full[s], 1);
      bars->n_sent[s] = 0;
    }
    mbar_init(&bars->lx, 256);
    mbar_init(&bars->fin_staged, 128);
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->acc_free, 16);
    mbar_init(&bars->epi_done, 8);
    item_ring_init(&bars->items, kItemReaders);
    mbar_init(&bars->mma_drain, 1);
    bars->abort_flag = 0;
    bars->fin_sent = 0;
    bars->n_recv = 0;
    bars->n_loaded = 0;
    bars->n_issued = 0;
    uint32_t sm;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
    bars->smid = sm < (uint32_t)kScratchSms ? (int)sm : -1;
    // an SM id outside the scratch: a capacity error, latched before the
    // abort it causes can latch a timeout
    if (bars->smid < 0) atomicCAS(p.status, 0, kStatusScratch);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&bars->tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // every CTA's barriers exist before any remote arrive, load or copy
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;

  auto get_item = [&](int k, bool& ok) { return item_get(&bars->items, k, ok, abort_flag, R); };
  auto get_item_warp = [&](int k, bool& ok) { return item_get_warp(&bars->items, k, ok, abort_flag, R, lane); };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA (both CTAs of a pair)
    if (elect_one()) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      int issued = 0;
      bool ok = true;
      const int nr = producer ? NR_P : NR_A;
      for (int k = 0; ok; ++k) {
        const int id = get_item(k, ok);
        if (id < 0) break;
        const FwdItem x = make_fwd_item(g, id, npairs, h);
        for (int n = 0; ok && n < x.N; ++n) {
          if (rank == 0 && n == x.N - 1) item_request(&bars->items);  // the next item is soon needed
          const int j0 = x.ks.tile(n) * T;
          for (int c = 0; c < 2; ++c, ++issued) {
            const int s = issued % nr;
            if (issued >= nr && !mbar_wait_cl(&bars->ring_empty[s], ((issued / nr) & 1) ^ 1, abort_flag, R)) {
              ok = false;
              break;
            }
            const uint32_t fb = mapa(smem_u32(&bars->ring_full[s]), lead);
            if (producer) {
              // this CTA's 64 keys, head-dim columns [256 c, 256 c + 256)
              if (leader) mbar_arrive_expect_tx(&bars->ring_full[s], 2 * SLOT_P);
              tma_load_4d_pair(base + OFF_RING_P + s * SLOT_P, &tmK, fb, 0, j0 + HT * (int)h, 4 * c, x.bkv);
            } else {
              // the 128 keys, this CTA's 128 columns of chunk c (head-dim columns [256 c + 128 h, +128))
              if (leader) mbar_arrive_expect_tx(&bars->ring_full[s], 2 * SLOT_A);
              tma_load_4d_pair(base + OFF_RING_A + s * SLOT_A, &tmV, fb, 0, j0, 4 * c + 2 * (int)h, x.bkv);
            }
          }
        }
        bars->n_issued = issued;
      }
      bars->n_issued = issued;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    if (elect_one()) {
      bool ok = true;
      if (producer) {
        const uint32_t idS = idesc_f16(2 * T, T, 1, 1, 0, 0);  // Q (TMEM) x K half (K-major), both bf16
        const uint64_t rd = smem_desc_sw128(sbase + OFF_RING_P, 16, 1024);
        const uint32_t x_tm = tmem + X_COL;
        int kp = 0, nc = 0;  // items, steps so far
        for (int k = 0; ok; ++k) {
          const int id = get_item(k, ok);
          if (id < 0) break;
          const FwdItem x = make_fwd_item(g, id, npairs, h);
          // both CTAs: the item's Q is in Tensor Memory -> tell the leader
          ok = mbar_wait_cl(&bars->q_ready, kp & 1, abort_flag, R);
          if (ok) {
            tc_fence_after();
            tc_fence_before();
            if (leader) mbar_arrive(&bars->pair_ready);
            else mbar_arrive_remote(mapa(smem_u32(&bars->pair_ready), lead));
          }
          if (leader && ok) ok = mbar_wait_cl(&bars->pair_ready, kp & 1, abort_flag, R);
          ++kp;
          if (!leader) continue;
          for (int n = 0; ok && n < x.N; ++n, ++nc) {
            const int bb = nc & 1;
            if (nc >= 2 && !mbar_wait_cl(&bars->s_free[bb], ((nc >> 1) - 1) & 1, abort_flag, R)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t s_tm = tmem + S_COL + bb * T;
            // unrolled over the step: constant operand offsets from a per-slot
            // base keep the single issuing thread ahead of the tensor pipe
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              const int li = 2 * nc + kk, s = li % NR_P;
              if (!mbar_wait_cl(&bars->ring_full[s], (li / NR_P) & 1, abort_flag, R)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t kd = rd + (uint64_t)(s * (SLOT_P >> 4));
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                  // head-dim columns 256 kk + 64 cc + 16 ks: Q columns 128 kk + 32 cc + 8 ks in TMEM
                  mma_pair_ts(s_tm, x_tm + 128 * kk + 32 * cc + 8 * ks, desc_add(kd, cc * HT * 128 + ks * 32), idS,
                              (kk | cc | ks) ? 1u : 0u);
                }
              }
              mma_commit_pair(&bars->ring_empty[s], pmask);
            }
            if (!ok) break;
            mma_commit_pair(&bars->s_full[bb], pmask);
          }
        }
      } else if (leader) {
        const uint32_t idPV = idesc_f16(2 * T, 256, 0, 0, 0, 1);  // P (K-major) x V half chunks (MN-major)
        int used = 0, nc = 0, ka = 0;  // ring loads consumed, steps, items so far
        for (int k = 0; ok; ++k) {
          const int id = get_item(k, ok);
          if (id < 0) break;
          const FwdItem x = make_fwd_item(g, id, npairs, h);
          // both CTAs' epilogues have read the previous item's O out of Tensor Memory
          if (ka > 0 && !mbar_wait_cl(&bars->acc_free, (ka - 1) & 1, abort_flag, R)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int n = 0; ok && n < x.N; ++n, ++nc) {
            const int bb = nc & 1;
            // both CTAs rescaled their rows, which they do once their P tile landed
            if (!mbar_wait_cl(&bars->o_ready[bb], (nc >> 1) & 1, abort_flag, R)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t ad = smem_desc_sw128(sbase + OFF_RECV + bb * TILE_BYTES, 16, 1024);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const int s = used % NR_A;
              if (!mbar_wait_cl(&bars->ring_full[s], (used / NR_A) & 1, abort_flag, R)) {
                ok = false;
                break;
              }
              ++used;
              tc_fence_after();
              const uint64_t vd = smem_desc_sw128(sbase + OFF_RING_A + s * SLOT_A, T * 128, 1024);
#pragma unroll
              for (int ks = 0; ks < T / 16; ++ks)
                mma_pair_ss(tmem + 256 * c, desc_add(ad, (ks >> 2) * T * 128 + (ks & 3) * 32),
                            desc_add(vd, ks * 2048), idPV, (n | ks) ? 1u : 0u);
              mma_commit_pair(&bars->ring_empty[s], pmask);
            }
            if (!ok) break;
            mma_commit_pair(&bars->mma_done[bb], pmask);
          }
          if (!ok) break;
          mma_commit_pair(&bars->acc_done, pmask);
          ++ka;
        }
      }
      // every MMA the leader issued has finished before either CTA releases Tensor Memory
      if (leader) mma_commit_pair(&bars->mma_drain, pmask);
      mbar_wait_drain(&bars->mma_drain, 0);
    }
  } else if (warp == kSigWarp) {
    if (rank == 0 && elect_one()) {
      // ---------------------------------------------------------- scheduler (rank 0)
      // items one at a time, drawn on rank 0's TMA thread's request
      // (cluster_items.cuh); a cluster that starts late or draws short
      // items takes more of them
      item_schedule(&bars->items, p.work, p.n_items, abort_flag, R);
    } else if (!producer && elect_one()) {
      // ---------------------------------------------------------- tile loads (accumulators)
      // once the MMAs of the step two steps back are done with the slot and
      // the producer's tile is in the scratch, load it (P tile, then its
      // factors); per item, arm the landing of its 1 / l
      const unsigned char* scr = g_fwd_tile_scratch + (size_t)(bars->smid < 0 ? 0 : bars->smid) * 2 * SCR_SLOT;
      bool ok = bars->smid >= 0;
      if (!ok) cluster_abort(abort_flag, R);
      int nc = 0, ka = 0;  // steps, items so far
      for (int k = 0; ok; ++k) {
        const int id = get_item(k, ok);
        if (id < 0) break;
        const FwdItem x = make_fwd_item(g, id, npairs, h);
        mbar_arrive_expect_tx(&bars->fin_full[ka & 1], 512);
        // the receive slots held the previous item's epilogue staging
        if (ka > 0 && !mbar_wait_cl(&bars->epi_done, (ka - 1) & 1, abort_flag, R)) {
          ok = false;
          break;
        }
        for (int n = 0; ok && n < x.N; ++n, ++nc) {
          const int bb = nc & 1;
          if (nc >= 2 && !mbar_wait_cl(&bars->mma_done[bb], ((nc >> 1) - 1) & 1, abort_flag, R)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->recv_full[bb], TILE_BYTES + 512);
          if (!mbar_wait_cl(&bars->tile_ready[bb], (nc >> 1) & 1, abort_flag, R)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
          bulk_load_g2s(sbase + OFF_RECV + bb * TILE_BYTES, scr + bb * SCR_SLOT, TILE_BYTES, &bars->recv_full[bb]);
          bulk_load_g2s(sbase + OFF_RVEC + bb * 512, scr + bb * SCR_SLOT + TILE_BYTES, 512, &bars->recv_full[bb]);
          bars->n_loaded = nc + 1;
        }
        ++ka;
      }
    } else if (producer && !leader && elect_one()) {
      // ---------------------------------------------------------- relay (producer peer)
      bool ok = true;
      int nc = 0;
      for (int k = 0; ok; ++k) {
        const int id = get_item(k, ok);
        if (id < 0) break;
        const FwdItem x = make_fwd_item(g, id, npairs, h);
        for (int n = 0; n < x.N; ++n, ++nc) {
          if (!mbar_wait_cl(&bars->s_free[nc & 1], (nc >> 1) & 1, abort_flag, R)) {
            ok = false;
            break;
          }
          mbar_arrive_remote(mapa(smem_u32(&bars->s_free[nc & 1]), lead));
        }
      }
    }
  } else if (warp == kRelayWarp) {
    if (producer && elect_one()) {
      // ---------------------------------------------------------- tile stores (producers)
      int sm_dst;
      asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(sm_dst) : "r"(mapa(smem_u32(&bars->smid), 2u + h))
                   : "memory");
      bool ok = sm_dst >= 0;
      if (!ok) cluster_abort(abort_flag, R);
      unsigned char* scr = g_fwd_tile_scratch + (size_t)(sm_dst < 0 ? 0 : sm_dst) * 2 * SCR_SLOT;
      int nc = 0;
      for (int k = 0; ok; ++k) {
        const int id = get_item(k, ok);
        if (id < 0) break;
        const FwdItem x = make_fwd_item(g, id, npairs, h);
        for (int n = 0; ok && n < x.N; ++n, ++nc) {
          const int bb = nc & 1;
          if (nc >= 2 && !mbar_wait_cl(&bars->scratch_free[bb], ((nc >> 1) - 1) & 1, abort_flag, R)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
          unsigned char* gdst = scr + bb * SCR_SLOT;
          for (int w = 0; w < 2; ++w) {
            // one barrier per staging tile: the warpgroups can be a step ahead of this warp
            if (!mbar_wait_cl(&bars->staged[bb][w], (nc >> 1) & 1, abort_flag, R)) {
              ok = false;
              break;
            }
            bulk_store_s2g(gdst + w * HALF_BYTES, sbase + OFF_STG + bb * TILE_BYTES + w * HALF_BYTES, HALF_BYTES);
          }
          if (!ok) break;
          bulk_store_s2g(gdst + TILE_BYTES, sbase + OFF_VEC + bb * 512, 512);  // the step's row factors
          bulk_commit_group();
          bulk_wait_read_all();
          mbar_arrive(&bars->stg_free[bb][0]);
          mbar_arrive(&bars->stg_free[bb][1]);
          bulk_wait_all();
          fence_proxy_async_global();
          mbar_arrive_remote(mapa(smem_u32(&bars->tile_ready[bb]), 2u + h));
        }
      }
      bulk_wait_all();  // no store still reads this CTA's shared memory
    }
    if (!producer && !leader && elect_one()) {
      // ---------------------------------------------------------- relay (accumulator peer)
      bool ok = true;
      int nc = 0;
      for (int k = 0; ok; ++k) {
        const int id = get_item(k, ok);
        if (id < 0) break;
        const FwdItem x = make_fwd_item(g, id, npairs, h);
        for (int n = 0; n < x.N; ++n, ++nc) {
          if (!mbar_wait_cl(&bars->o_ready[nc & 1], (nc >> 1) & 1, abort_flag, R)) {
            ok = false;
            break;
          }
          mbar_arrive_remote(mapa(smem_u32(&bars->o_ready[nc & 1]), lead));
        }
      }
    }
  } else if (producer) {
    // ------------------------------------------------------------ softmax (producers, both CTAs)
    const int wg = (warp - 2) >> 2, q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const int cb0 = 64 * wg;
    const float sl2 = g.scale * kLog2e;
    float* alph = reinterpret_cast<float*>(base + OFF_VEC);  // [2 tile][128]
    float* xm = alph + 384;                                   // [2 parity][2 wg][128]
    float* xl = xm + 512;                                     // [2 wg][128]
    float* finl = xl + 256;                                   // [2 item parity][128]
    const uint32_t acc = 2u + h;                              // accumulator CTA of this half
    const uint32_t stg0 = sbase + OFF_STG + wg * HALF_BYTES;
    const bool issuer = (warp & 3) == 2;  // warp 2 / 6 copies its warpgroup's half
    bool ok = true;
    int nc = 0, kp = 0;  // steps, items so far
    for (int k = 0; ok; ++k) {
      const int id = get_item_warp(k, ok);
      if (id < 0) break;
      const FwdItem x = make_fwd_item(g, id, npairs, h);
      const int i = x.i0 + r;
      const bool row_ok = i < g.Lq;
      {
        // Q row i into Tensor Memory: bf16 pairs, one 32-bit column each;
        // warpgroup wg fills columns [128 wg, 128 wg + 128) (head-dim elements
        // [256 wg, 256 wg + 256)).  The previous item's S MMAs, the only
        // readers, finished: their s_full was seen before its last S was read.
        const uint4* src =
            reinterpret_cast<const uint4*>(p.q + ((size_t)x.bh * g.Lq + (row_ok ? i : 0)) * DH) + wg * 32;
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          uint32_t v[32];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint4 w4 = row_ok ? __ldg(src + j * 8 + q) : make_uint4(0u, 0u, 0u, 0u);
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
      float m_run = -INFINITY, l_run = 0.f;
      for (int n = 0; n < x.N; ++n, ++nc) {
        const int bb = nc & 1;
        const int j0 = x.ks.tile(n) * T;
        if (!__all_sync(0xffffffffu, mbar_wait_cl(&bars->s_full[bb], (nc >> 1) & 1, abort_flag, R))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld32(tmem + lane_off + S_COL + bb * T + cb0, *reinterpret_cast<uint32_t(*)[32]>(sr));
        tmem_ld32(tmem + lane_off + S_COL + bb * T + cb0 + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_free[bb]);  // the peer's relay tells the leader
        const bool full = x.own_rows && rows_tile_full(g, x.i0, x.ihi, j0, j0 + T - 1);
        // visible key columns of row i in this tile, relative to this warpgroup's half
        bool both;
        const int4 vv = vis_in_tile(row_vis(g, i, j0 + cb0), 64, &both);
        const bool two_here = two && __any_sync(0xffffffffu, both);
        float pmax;
        if (sl2 > 0.f)
          pmax = sl2 * (full ? half_max_raw<true>(sr, vv)
                             : (two_here ? half_max_raw<false, true>(sr, vv) : half_max_raw<false>(sr, vv)));
        else
          pmax = full ? half_max<true>(sr, sl2, vv)
                      : (two_here ? half_max<false, true>(sr, sl2, vv) : half_max<false>(sr, sl2, vv));
        // the two warps of this lane quarter exchange their halves' maxima
        xm[(bb * 2 + wg) * 128 + r] = pmax;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->mx[bb][q4]);
        if (!__all_sync(0xffffffffu, mbar_wait_cl(&bars->mx[bb][q4], (nc >> 1) & 1, abort_flag, R))) {
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
        const float tsum = full ? half_p<true>(sr, sl2, m_use, vv, pk)
                                : (two_here ? half_p<false, true>(sr, sl2, m_use, vv, pk)
                                            : half_p<false>(sr, sl2, m_use, vv, pk));
        l_run = l_run * alpha + tsum;
        // the store of this staging half two steps ago (and of that alpha) must have read it
        if (nc >= 2 &&
            !__all_sync(0xffffffffu, mbar_wait_cl(&bars->stg_free[bb][wg], ((nc >> 1) - 1) & 1, abort_flag, R))) {
          ok = false;
          break;
        }
        const uint32_t stg = stg0 + bb * TILE_BYTES;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          st_smem_v4(stg + r * 128 + ((u ^ (r & 7)) << 4), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        if (wg == 0) alph[bb * 128 + r] = alpha;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->staged[bb][wg]);  // the store warp takes the tile from here
        bars->n_sent[wg] = nc + 1;
      }
      if (!ok) break;
      // row sum = the two warpgroups' partial sums (same running max); lse; send 1 / l
      xl[wg * 128 + r] = l_run;
      mbar_arrive(&bars->lx);
      if (!__all_sync(0xffffffffu, mbar_wait_cl(&bars->lx, kp & 1, abort_flag, R))) {
        ok = false;
        break;
      }
      const float l_tot = xl[r] + xl[128 + r];
      if (wg == 0) {
        // 1 / l, or with attention sinks the factor that folds the head's
        // sink logit into the row's normaliser; the accumulator scales O by
        // it.  Two buffers by item parity: the copy of the previous item's
        // factors may still be reading the other one.
        float lse_row = (m_run + log2f(l_tot)) * kLn2;
        float fin = 1.f / l_tot;
        if (g.sinks) fin = sink_finish(g.sinks[x.bh % g.Hq], m_run, l_tot, &lse_row);
        if (row_ok) p.lse[(size_t)x.bh * g.Lq + i] = lse_row;
        float* fl = finl + (kp & 1) * 128;
        fl[r] = fin;
        fence_proxy_async_smem();
        mbar_arrive(&bars->fin_staged);
        if (issuer && __all_sync(0xffffffffu, mbar_wait_cl(&bars->fin_staged, kp & 1, abort_flag, R)) && lane == 0) {
          bulk_copy_to_cta(mapa(sbase + OFF_RVEC + 1024 + (uint32_t)(kp & 1) * 512u, acc), smem_u32(fl), 512,
                           mapa(smem_u32(&bars->fin_full[kp & 1]), acc));
          bars->fin_sent = kp + 1;
        }
      }
      ++kp;
    }
    // (unwinding: the store warp waits for its own stores)
  } else {
    // ------------------------------------------------------------ rescale + epilogue (accumulators, both CTAs)
    const int wg = (warp - 2) >> 2, q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const float* ralph = reinterpret_cast<const float*>(base + OFF_RVEC);  // [2][128]
    const float* rinv = ralph + 256;                                       // [2 item parity][128]
    bool ok = true;
    int nc = 0, ka = 0;  // steps, items so far
    for (int k = 0; ok; ++k) {
      const int id = get_item_warp(k, ok);
      if (id < 0) break;
      const FwdItem x = make_fwd_item(g, id, npairs, h);
      for (int n = 0; n < x.N; ++n, ++nc) {
        const int bb = nc & 1;
        if (!__all_sync(0xffffffffu, mbar_wait_cl(&bars->recv_full[bb], (nc >> 1) & 1, abort_flag, R))) {
          ok = false;
          break;
        }
        if (threadIdx.x == 64) {
          bars->n_recv = nc + 1;
          // the producer may store its next tile into this scratch slot
          mbar_arrive_remote(mapa(smem_u32(&bars->scratch_free[bb]), h));
        }
        const float a = ralph[bb * 128 + r];
        if (__any_sync(0xffffffffu, a != 1.f)) {
          // O must hold PV of every earlier step of the item before it is
          // rescaled (the first step's factor is always 1)
          if (n >= 1 && !__all_sync(0xffffffffu, mbar_wait_cl(&bars->mma_done[(nc - 1) & 1], ((nc - 1) >> 1) & 1,
                                                               abort_flag, R))) {
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
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->o_ready[bb]);  // the peer's relay tells the leader
      }
      if (!ok) break;
      if (!__all_sync(0xffffffffu, mbar_wait_cl(&bars->acc_done, ka & 1, abort_flag, R) &&
                                       mbar_wait_cl(&bars->fin_full[ka & 1], (ka >> 1) & 1, abort_flag, R))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float inv = rinv[(ka & 1) * 128 + r];
      // the receive slots have been consumed by the finished MMAs, and the
      // tile loads wait for epi_done: each of warps 2-9 stages its O blocks
      // in two 4 KB buffers there (the V ring may already hold the next
      // item's loads)
      tmem_rows_store_tma<2, false>(&tmO, tmem + lane_off + 256 * wg, 256 * wg, 256, inv,
                                    sbase + OFF_RECV + (uint32_t)(warp - 2) * 8192u, x.i0 + 32 * q4, x.bh, lane);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars->epi_done);  // the staging may be overwritten
        // O may be overwritten
        if (leader) mbar_arrive(&bars->acc_free);
        else mbar_arrive_remote(mapa(smem_u32(&bars->acc_free), lead));
      }
      ++ka;
    }
    if (lane == 0) bulk_wait_all();  // the epilogue stores have written
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA issues a load, a copy or a remote arrival past this point
  if (threadIdx.x == 0 && *abort_flag) {
    // unwinding only.  Accumulators: tiles the producer of this half sent
    // that never landed, and its last 1 / l, must land before this CTA's
    // shared memory is released.
    if (!producer) {
      int fsent;
      asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(fsent) : "r"(mapa(smem_u32(&bars->fin_sent), h)) : "memory");
      for (int m = bars->n_recv; m < bars->n_loaded; ++m) mbar_wait_drain(&bars->recv_full[m & 1], (m >> 1) & 1);
      if (fsent > 0) mbar_wait_drain(&bars->fin_full[(fsent - 1) & 1], ((fsent - 1) >> 1) & 1);
    }
    // Leader: the ring loads of both CTAs complete on its barriers; let the
    // last load of each slot (of either CTA) land.
    if (leader) {
      int peer_issued;
      asm volatile("ld.shared::cluster.u32 %0, [%1];"
                   : "=r"(peer_issued)
                   : "r"(mapa(smem_u32(&bars->n_issued), lead + 1))
                   : "memory");
      const int issued = max(bars->n_issued, peer_issued);
      const int nr = producer ? NR_P : NR_A;
      for (int k = issued - 1; k >= 0 && k >= issued - nr; --k)
        mbar_wait_drain(&bars->ring_full[k % nr], (k / nr) & 1);
    }
  }
  __syncthreads();
  cluster_sync();
  if (*abort_flag && threadIdx.x == 0) atomicCAS(p.status, 0, kStatusTimeout);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// Clusters that fit on the current device at once (cached per device; 0 on
// an error).
int max_clusters(const cudaLaunchConfig_t& cfg) {
  static std::atomic<int> cached[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < kMaxDevices) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fwd512_kernel, &cfg) != cudaSuccess) return 0;
  if (dev < kMaxDevices && n > 0) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace

int scratch_layout_fwd512() {
  int n = 0, nsm = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev))
    return -1;
  if (cudaFuncSetAttribute(fwd512_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM) ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fwd512_kernel, kThr, SMEM))
    return -1;
  return (n == 1 && nsm <= kScratchSms) ? 0 : 1;
}

cudaError_t launch_fwd_tc512(const Geom& g, const uint16_t* q, const uint16_t* k, const uint16_t* v16, float* o,
                             float* lse, int* work, int* status, cudaStream_t s) {
  if (!work) return cudaErrorInvalidValue;
  CUtensorMap tk, tv, to;
  cudaError_t e;
  // K: 64 keys x four 64-column chunks per instruction (32 KB, one CTA's half
  // of a 256-column slice); V: 128 keys x two chunks (32 KB)
  if ((e = make_tmap_f16_chunks(&tk, k, DH, g.L, g.B * g.Hkv, HT, 4)) != cudaSuccess) return e;
  if ((e = make_tmap_f16_chunks(&tv, v16, DH, g.L, g.B * g.Hkv, T, 2)) != cudaSuccess) return e;
  if ((e = make_tmap_f32_out(&to, o, DH, g.Lq, g.B * g.Hq)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(fwd512_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM)) !=
      cudaSuccess)
    return e;
  FwdPairParams pm;
  pm.g = g;
  pm.q = q;
  pm.o = o;
  pm.lse = lse;
  pm.n_tiles = (g.Lq + T - 1) / T;
  pm.work = work;
  pm.n_items = g.B * g.Hkv * ((pm.n_tiles + 1) / 2) * g.G;
  pm.status = status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(R, 1, 1);
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
  // persistent clusters: as many as fit on the GPU at once, at most one per item
  const int fit = max_clusters(cfg);
  if (fit <= 0) return cudaErrorInvalidConfiguration;
  cfg.gridDim = dim3(R * (unsigned)min(fit, pm.n_items), 1, 1);
  return cudaLaunchKernelEx(&cfg, fwd512_kernel, tk, tv, to, pm);
}

}  // namespace swa
