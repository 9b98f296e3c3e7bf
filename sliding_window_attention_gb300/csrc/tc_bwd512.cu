// Tensor-core backward for head dim 512 on clusters of CTA pairs.
//
// At D = 512 the two accumulators of a 128-key tile (dK and dV, 512 fp32
// columns each) need twice the Tensor Memory of one SM, and K plus V of the
// tile (128 KB each in fp16) do not fit one SM's shared memory together.  So
// the work is split by role across the CTAs of a cluster, and every role runs
// on a CTA pair (tcgen05 .cta_group::2): the pair owns two adjacent 128-row
// tiles of the resident side (keys in the dK/dV pass, queries in the dQ
// pass), one per CTA, and each MMA of M = 256 rows takes its B operand half
// from each CTA.  Every streamed tile therefore crosses each SM's TMA engine
// and shared memory only once per pair, half in each CTA.
//   producers (three pairs in the dK/dV pass, ranks 0-5, two in the dQ
//     pass, ranks 0-3, taking the streamed steps in turn): the A operand of S (K for dK/dV, Q for dQ: 128 x 512 fp16 per
//     CTA = 256 columns) lives in Tensor Memory and feeds TS-form MMAs, the A
//     operand of dP (V, or dO) in shared memory; the streamed tile arrives as
//     two 64-row halves, one per CTA, in 16 KB slices of 128 columns.  Each
//     CTA forms S and dP for its 128 rows and all 128 streamed columns, then
//     P = exp(scale S - lse) and dS = P (dP - Delta) ("Training -- design
//     (ORPO, flash-CCE head, prefix sharing, segmented backward)", section 6:
//     recompute P from the stored lse), and hands the fp16 tiles to the
//     accumulator CTA of the same half through an L2 scratch (below);
//   accumulators (one pair per accumulator: ranks 6-7 dV += P^T dO and 8-9
//     dK += dS^T Q in the dK/dV pass, ranks 4-5 dQ += dS K in the dQ pass)
//     hold one 128 x 512 fp32 accumulator per CTA in Tensor Memory; the
//     streamed operand arrives in 128-column halves of 256-column chunks and
//     each step is 16 MMAs of M = 256, N = 256.
// Only tiles that meet the causal / window band are visited ("Lab 028 lab
// detail: Off NVIDIA, you fix the platform yourself", "What I changed, in
// plain terms" items 3-4); the two tiles of a pair walk the union of their
// bands, and the columns outside a row's band are zero in P and dS.
//
// Warps: 0 TMA, 1 Tensor Memory owner and (leader CTA) MMA issuer, 2-9
// elementwise (two warpgroups, 64 of the 128 columns each: producers stage
// their half of each tile; in accumulators warps 2 .. 1 + NPP watch the
// tiles land and the next NPP warps load them, one warp per producer pair,
// before all of 2-9 write the result), 10 relay of the peer's releases
// (producer peers) or the work-item scheduler (rank 0), 11 tile stores
// (producers).  Both passes are persistent: as many clusters as fit on the
// GPU loop over work items (cluster_items.cuh), the next item's resident
// operands loading while the accumulators finish the previous one; the dQ
// pass starts beside the dK/dV pass as a programmatic dependent launch.
// Every wait is bounded; a timeout in one CTA is broadcast to
// the whole cluster, every CTA drains its loads, stores and MMAs in flight,
// and the status word records the timeout.
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

constexpr int kDirKV = 0, kDirQ = 1;
constexpr int kMaxDevices = 64;
constexpr int kRoleProd = 0, kRoleAccP = 1, kRoleAccDS = 2;
constexpr int T = 128;     // rows of a resident tile, columns of a streamed step
constexpr int HT = 64;     // streamed rows per CTA of a pair
constexpr int DH = 512;    // head dim
constexpr int kThr = 384;  // 12 warps
constexpr int kSigWarp = 10;
constexpr int kStoreWarp = 11;
constexpr float kLog2e = 1.4426950408889634f;

constexpr int RES_BYTES = T * DH * 2;       // resident dP A operand (V or dO), fp16
constexpr int TILE_BYTES = T * T * 2;       // fp16 128 x 128 operand tile
constexpr int HALF_BYTES = TILE_BYTES / 2;  // one warpgroup's 64-column half (one swizzle chunk)
// producer: resident operand, two staging halves, ring of 16 KB slices (two
// 64-column chunks of this CTA's 64 streamed rows)
constexpr int NR_P = 4;
constexpr int SLOT_P = 2 * HT * 128;
constexpr int OFF_STG = RES_BYTES;
constexpr int OFF_RING_P = RES_BYTES + 2 * HALF_BYTES;
constexpr int DATA_BYTES = OFF_RING_P + NR_P * SLOT_P;
// Per pass: NPP producer pairs take the streamed steps in turn.  The dK/dV
// pass has two accumulator pairs to feed per step and three producer pairs
// (10-CTA clusters); the dQ pass has one accumulator pair and two producer
// pairs (6-CTA clusters).  An accumulator holds RS operand slots per producer
// pair (with two, a producer can send its next tile while the accumulator
// still works on the previous one), then a ring of 32 KB slots (two 64-column
// chunks of the 128 streamed rows).
constexpr int OFF_RECV = 0;
constexpr int SLOT_A = 2 * T * 128;
template <int DIR>
struct PassCfg {
  static constexpr int NPP = DIR == kDirKV ? 3 : 2;
  static constexpr int RS = DIR == kDirKV ? 1 : 2;
  static constexpr int NRECV = NPP * RS;
  static constexpr uint32_t R = 2 * NPP + (DIR == kDirKV ? 4 : 2);  // CTAs per cluster
  static constexpr int OFF_RING_A = NRECV * TILE_BYTES;
  static constexpr int NR_A = (DATA_BYTES - OFF_RING_A) / SLOT_A;
  static_assert(NR_A >= 2 && OFF_RING_A + NR_A * SLOT_A <= DATA_BYTES, "accumulator footprint");
};
constexpr int kMaxNpp = 3, kMaxRs = 2, kMaxRecv = 4;
constexpr int kMaxRing = 4;
static_assert(PassCfg<kDirKV>::NRECV <= kMaxRecv && PassCfg<kDirQ>::NRECV <= kMaxRecv, "receive slots");
static_assert(PassCfg<kDirKV>::NR_A <= kMaxRing && PassCfg<kDirQ>::NR_A <= kMaxRing && NR_P <= kMaxRing, "rings");
// producer, dK/dV pass: each warpgroup's step statistics (lse * log2e and
// Delta of its 64 columns) staged in shared memory
constexpr int OFF_STATS = DATA_BYTES;
constexpr int STATS_BYTES = 2 * 512;
// producer Tensor Memory: resident S operand (fp16 pairs), S, dP
constexpr uint32_t X_COL = 0, S_COL = 256, DP_COL = 384;

// Producer -> accumulator tiles travel through L2: the producer bulk-stores
// a staged tile into the scratch of the accumulator CTA's SM (its staging is
// free again as soon as the store has read it) and the accumulator loads it
// into its operand slot.  One CTA of these kernels fills an SM, so the
// scratch of an SM belongs to one accumulator CTA at a time, whichever pass
// it belongs to (the two passes run side by side): kMaxRecv slots of two
// 16 KB halves per SM, of which a pass uses its NRECV.
constexpr int kScratchSms = 192;
__device__ __align__(1024) unsigned char g_tile_scratch[(size_t)kScratchSms * kMaxRecv * TILE_BYTES];

struct Bars {
  uint64_t res_full;              // (leader) both CTAs' resident dP operand landed
  uint64_t x_ready;               // (own) resident S operand written to Tensor Memory
  uint64_t pair_ready;            // (leader) both CTAs' resident S operand ready
  uint64_t ring_full[kMaxRing];   // (leader) both halves of a ring slot landed
  uint64_t ring_empty[kMaxRing];  // (both) the pair's MMAs finished reading a slot
  uint64_t s_full, p_full;        // (producer, both) S / dP of a step in Tensor Memory
  uint64_t s_free, p_free;        // (producer) S / dP read: leader counts its 8 warps and the peer's relay
  uint64_t staged[2];             // (producer) a warpgroup wrote its staging half
  uint64_t stg_free[2];           // (producer) the store thread has read a staging half out
  uint64_t scratch_free[2][kMaxRs];  // (producer) the accumulator loaded the scratch slot: [0] P -> dV, [1] dS -> dK / dQ
  uint64_t stats_full[2];         // (producer, dK/dV) a warpgroup's step statistics landed
  uint64_t stats_free[2];         // (producer, dK/dV) a warpgroup read its step statistics
  uint64_t tile_ready[kMaxRecv];     // (accumulator) the producer's tile for slot is in the scratch
  uint64_t recv_full[kMaxRecv][2];   // (accumulator, own) half of the tile loaded into slot
  uint64_t peer_recv[kMaxRecv];      // (accumulator leader) the peer's tile landed in slot
  uint64_t mma_done[kMaxRecv];       // (accumulator, both) MMAs reading slot finished
  uint64_t acc_done;                 // (accumulator, both) an item's MMAs finished
  uint64_t acc_free;                 // (accumulator leader) both CTAs read an item's accumulator out
  uint64_t epi_done;                 // (accumulator, own) the epilogue's stores read their staging
  uint64_t mma_drain;
  uint32_t tmem_slot;
  int abort_flag;
  int smid;                       // (accumulator) SM this CTA runs on: the scratch it loads from
  int n_loaded[kMaxNpp];          // (accumulator) own steps of producer pair p whose loads were issued
  int n_recv[kMaxNpp];            // (accumulator) own steps of producer pair p observed landed
  int n_issued;                   // ring loads issued by this CTA
  int n_res;                      // (producer) resident loads issued by this CTA
  ItemRing items;                // work-item ids from rank 0's scheduler
};

constexpr size_t SMEM = (size_t)DATA_BYTES + STATS_BYTES + 1024 + 1024;
static_assert(SMEM <= 232448, "shared memory");
static_assert(sizeof(Bars) <= 1024, "barrier block");

struct ParamsPair {
  Geom g;
  int* work;            // the pass's work counter: the next item id (zero before the launch)
  int n_items;          // work items
  float* out0;          // KV: dk ; Q: dq
  float* out1;          // KV: dv
  const uint16_t* x16;  // resident S operand rows: KV: k16 ; Q: q16
  const float* stats;   // two planes: lse * log2e, then Delta (B * Hq * Lpad floats each)
  int Lpad;
  int n_tiles;          // resident-side 128-row tiles
  int* status;
};

// P for 64 columns (cb0 .. cb0 + 63 of the tile) of one row, in place over the
// S values (fp32).  PER_COL: the lse belongs to the column (lse_s is the
// shared address of lse * log2e of the 64 columns); otherwise l2 is the row's.
// Columns outside the row's visible columns v (tile-local; see vis(), TWO
// under a shared-prefix plan) are exactly zero unless FULL.
template <bool FULL, bool PER_COL, bool TWO = false>
__device__ __forceinline__ void p_tile64(uint32_t (&sv)[64], uint32_t lse_s, float l2, float sl2, int cb0,
                                         const int4& v) {
#pragma unroll
  for (int e = 0; e < 64; e += 4) {
    float lv[4] = {l2, l2, l2, l2};
    if (PER_COL) {
      const float4 l4 = ld_smem_f4(lse_s + 4 * e);
      lv[0] = l4.x;
      lv[1] = l4.y;
      lv[2] = l4.z;
      lv[3] = l4.w;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float pv = fast_exp2(fmaf(__uint_as_float(sv[e + u]), sl2, -lv[u]));
      if (!FULL) pv = vis<TWO>(cb0 + e + u, v) ? pv : 0.f;
      sv[e + u] = __float_as_uint(pv);
    }
  }
}

__device__ __forceinline__ void pack64(const uint32_t (&v)[64], uint32_t (&o)[32]) {
#pragma unroll
  for (int e = 0; e < 64; e += 2) o[e >> 1] = pack_half2(__uint_as_float(v[e]), __uint_as_float(v[e + 1]));
}

// dS = P (dP - Delta) for 64 columns as fp16 pairs (dl_s: shared address of
// the Delta of the 64 columns when PER_COL; otherwise dl is the row's).
template <bool PER_COL>
__device__ __forceinline__ void ds_tile64(const uint32_t (&pv)[64], const uint32_t (&dv)[64], uint32_t dl_s,
                                          float dl, uint32_t (&o)[32]) {
#pragma unroll
  for (int e = 0; e < 64; e += 4) {
    float dd[4] = {dl, dl, dl, dl};
    if (PER_COL) {
      const float4 d4 = ld_smem_f4(dl_s + 4 * e);
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

// Arrive on `bar` of the pair's leader CTA (locally when this CTA is the leader).
__device__ __forceinline__ void arrive_leader(uint64_t* bar, bool leader, uint32_t lead) {
  if (leader) mbar_arrive(bar);
  else mbar_arrive_remote(mapa(smem_u32(bar), lead));
}

// One work item of a persistent cluster: a pair of resident-side tiles (keys
// in the dK/dV pass; in the dQ pass the query rows of one query head).  Ids
// run with the kv head (b * Hkv + kv head) slowest, then the tile pair (the
// longest band first), then (dQ pass) the group's query head, so that the
// clusters working at any moment share one kv head: its K and V (dQ pass) or
// its group's Q and dO (dK/dV pass) are read from HBM about once and then
// served by L2, and the short items come last.
struct Item {
  int bkv, b;       // b * Hkv + kv head, batch
  int head;         // head of the resident rows: kv head (dK/dV) or query head (dQ), batch included
  int pr0, prlast;  // first and last resident row of the pair
  int r0, rlast;    // this CTA's tile (rlast = r0 when it has no rows)
  bool own_rows;    // false for the second tile of an odd last pair
  TileSteps ts;     // dK/dV: the query tiles that can see a key of the pair; dQ: the key tiles meeting its band
  int ntq, N;       // streamed tiles; steps (dK/dV: tiles x the group's query heads)
};

template <int DIR>
__device__ __forceinline__ Item make_item(const Geom& g, int id, int npairs, int LX, uint32_t h) {
  Item x;
  const int per_kv = DIR == kDirKV ? npairs : npairs * g.G;
  x.bkv = id / per_kv;
  const int rem = id - x.bkv * per_kv;
  x.b = x.bkv / g.Hkv;
  int tp;
  if (DIR == kDirKV) {
    tp = rem;  // key tile pair 0 is seen by the most queries
    x.head = x.bkv;
  } else {
    const int y = rem / g.G;
    tp = npairs - 1 - y;  // the last query tile pair has the longest band
    x.head = x.b * g.Hq + (x.bkv - x.b * g.Hkv) * g.G + (rem - y * g.G);
  }
  x.pr0 = 2 * tp * T;
  x.prlast = min(x.pr0 + 2 * T, LX) - 1;
  x.r0 = x.pr0 + (int)h * T;
  x.own_rows = x.r0 < LX;
  x.rlast = x.own_rows ? min(x.r0 + T, LX) - 1 : x.r0;
  x.ts = DIR == kDirKV ? key_steps(g, x.pr0, x.prlast, T) : row_steps(g, x.pr0, x.prlast, T);
  x.ntq = x.ts.count();
  x.N = DIR == kDirKV ? g.G * x.ntq : x.ntq;
  return x;
}
// Streamed-side rows and head of step n of item x.  dK/dV pass: query tiles
// from the last one down, the group's query heads innermost, so that
// concurrent clusters of one kv head read the same Q and dO tiles at about
// the same time.
template <int DIR>
__device__ __forceinline__ int step_rows(const Geom& g, const Item& x, int n) {
  if (DIR == kDirKV) return x.ts.tile(x.ntq - 1 - n / g.G) * T;
  return x.ts.tile(n) * T;
}
template <int DIR>
__device__ __forceinline__ int step_head(const Geom& g, const Item& x, int n) {
  if (DIR == kDirKV) return x.b * g.Hq + (x.head - x.b * g.Hkv) * g.G + n % g.G;  // query head
  return x.bkv;                                                                  // kv head
}
// Producer pair pp takes steps pp, pp + NPP, ... of an item's N; its m-th
// own step is pp + NPP m.
template <int NPP>
__device__ __forceinline__ int own_steps(int N, int pp) {
  return max(0, (N - pp + NPP - 1) / NPP);
}
// Readers of each item id in a cluster (the scheduler counts their arrivals
// before it reuses the id's slot): per producer pair the leader's TMA, MMA,
// eight elementwise and store warps (11) and the peer's same plus its relay
// warp (12); per accumulator pair the leader's TMA, MMA and eight elementwise
// warps (10) and the peer's TMA and eight elementwise warps (9).
template <int DIR>
constexpr int item_readers() {
  return PassCfg<DIR>::NPP * (11 + 12) + (DIR == kDirKV ? 2 : 1) * (10 + 9);
}

template <int DIR>
__global__ void __launch_bounds__(kThr, 1)
    bwd512_kernel(const __grid_constant__ CUtensorMap tmS,   // streamed S operand, 64 rows x 2 chunks: Q / K
                   const __grid_constant__ CUtensorMap tmP,   // streamed dP operand, 64 rows x 2 chunks: dO / V
                   const __grid_constant__ CUtensorMap tmR,   // resident dP operand, 128 rows x 1 chunk: V / dO
                   const __grid_constant__ CUtensorMap tmA0,  // dV accumulator operand, 128 rows x 2 chunks: dO
                   const __grid_constant__ CUtensorMap tmA1,  // dK / dQ accumulator operand: Q / K
                   const __grid_constant__ CUtensorMap tmO0,  // fp32 output out0 (dk / dq), 32 x 32 boxes
                   const __grid_constant__ CUtensorMap tmO1,  // fp32 output out1 (dv; dQ pass: out0 again)
                   const ParamsPair p) {
  using C = PassCfg<DIR>;
  constexpr int NPP = C::NPP, RS = C::RS, NRECV = C::NRECV, NR_A = C::NR_A, OFF_RING_A = C::OFF_RING_A;
  constexpr uint32_t R = C::R;
  // cluster ranks: producers 0 .. 2 NPP - 1, then the accumulator pairs (dV,
  // then dK, in the dK/dV pass; dQ in the dQ pass)
  constexpr uint32_t kAccP = 2 * NPP, kAccDS = 2 * NPP + (DIR == kDirKV ? 2 : 0);
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(base + DATA_BYTES + STATS_BYTES);
  volatile int* abort_flag = &bars->abort_flag;
  const uint32_t sbase = smem_u32(base);

  const Geom& g = p.g;
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const uint32_t h = rank & 1u;      // half of the pair: which resident tile, which streamed rows
  const uint32_t lead = rank & ~1u;  // the pair's leader
  const bool leader = h == 0;
  const uint16_t pmask = (uint16_t)(3u << lead);
  const int role = rank < kAccP ? kRoleProd : ((DIR == kDirKV && rank < kAccDS) ? kRoleAccP : kRoleAccDS);
  const bool acc_role = role != kRoleProd;
  const int pp = (int)(rank >> 1);  // producer pair (producers only)
  const int LX = (DIR == kDirKV) ? g.L : g.Lq;  // rows of the resident side
  const int npairs = (p.n_tiles + 1) / 2;
  const bool two = g.Rc > 0;  // shared-prefix plan: two visible intervals per row
  // accumulator: which of the producer's two destinations this CTA is
  const int dst_kind = (role == kRoleAccP) ? 0 : 1;
  // the dQ pass, launched right after this one on the same stream, may start
  // on the SMs this pass leaves once all of its clusters are resident
  if (DIR == kDirKV && threadIdx.x == 0) grid_launch_dependents();

  if (threadIdx.x == 0) {
    mbar_init(&bars->res_full, 1);
    mbar_init(&bars->x_ready, 256);
    mbar_init(&bars->pair_ready, 2);
    for (int s = 0; s < kMaxRing; ++s) {
      mbar_init(&bars->ring_full[s], 1);
      mbar_init(&bars->ring_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->p_full, 1);
    // 8 elementwise warps, plus (leader) the one arrival the peer's relay warp forwards
    mbar_init(&bars->s_free, leader ? 9 : 8);
    mbar_init(&bars->p_free, leader ? 9 : 8);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->staged[s], 128);
      mbar_init(&bars->stg_free[s], 1);
      for (int j = 0; j < RS; ++j) mbar_init(&bars->scratch_free[s][j], 1);
      mbar_init(&bars->stats_full[s], 1);
      mbar_init(&bars->stats_free[s], 128);
    }
    item_ring_init(&bars->items, item_readers<DIR>());
    for (int s = 0; s < NRECV; ++s) {
      mbar_init(&bars->tile_ready[s], 1);
      mbar_init(&bars->recv_full[s][0], 1);
      mbar_init(&bars->recv_full[s][1], 1);
      mbar_init(&bars->peer_recv[s], 1);
      mbar_init(&bars->mma_done[s], 1);
    }
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->acc_free, 16);
    mbar_init(&bars->epi_done, 8);
    mbar_init(&bars->mma_drain, 1);
    bars->abort_flag = 0;
    uint32_t sm;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
    bars->smid = sm < (uint32_t)kScratchSms ? (int)sm : -1;
    // an SM id outside the scratch: a capacity error, latched before the
    // abort it causes can latch a timeout
    if (bars->smid < 0) atomicCAS(p.status, 0, kStatusScratch);
    for (int s = 0; s < NPP; ++s) bars->n_recv[s] = bars->n_loaded[s] = 0;
    bars->n_issued = 0;
    bars->n_res = 0;
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
      prefetch_tmap(&tmS);
      prefetch_tmap(&tmP);
      prefetch_tmap(&tmR);
      prefetch_tmap(&tmA0);
      prefetch_tmap(&tmA1);
      int issued = 0;  // ring loads issued
      int n_res = 0;   // producer: items with own steps so far
      int M = 0;       // producer: own steps so far
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int id = get_item(k, ok);
        if (id < 0) break;
        const Item x = make_item<DIR>(g, id, npairs, LX, h);
        if (!acc_role) {
          // resident dP operand (this CTA's 128 rows), then per own step four
          // slices for S and then four for dP (this CTA's 64 rows)
          const int n_own = own_steps<NPP>(x.N, pp);
          if (n_own == 0) {
            if (rank == 0) item_request(&bars->items);
            continue;
          }
          // the previous item's last dP has finished reading the resident operand
          if (n_res > 0 && !mbar_wait_cl(&bars->p_full, (M - 1) & 1, abort_flag, R)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&bars->res_full, 2 * RES_BYTES);
          const uint32_t res_bar = mapa(smem_u32(&bars->res_full), lead);
          for (int c = 0; c < DH / 64; ++c) tma_load_3d_pair(base + c * T * 128, &tmR, res_bar, c * 64, x.r0, x.head);
          bars->n_res = ++n_res;
          for (int m = 0; ok && m < n_own; ++m) {
            const int n = pp + NPP * m;
            const int rows = step_rows<DIR>(g, x, n) + HT * (int)h, hd = step_head<DIR>(g, x, n);
            if (rank == 0 && m == n_own - 1) item_request(&bars->items);  // the next item is soon needed
            for (int kk = 0; kk < 2 * (DH / 128); ++kk, ++issued) {
              const int s = issued % NR_P;
              if (issued >= NR_P && !mbar_wait_cl(&bars->ring_empty[s], ((issued / NR_P) & 1) ^ 1, abort_flag, R)) {
                ok = false;
                break;
              }
              if (leader) mbar_arrive_expect_tx(&bars->ring_full[s], 2 * SLOT_P);
              tma_load_4d_pair(base + OFF_RING_P + s * SLOT_P, kk >= 4 ? &tmP : &tmS,
                               mapa(smem_u32(&bars->ring_full[s]), lead), 0, rows, 2 * (kk & 3), hd);
            }
          }
          M += n_own;
        } else {
          // this CTA's 128-column half of each 256-column chunk of dO (dV), Q (dK) or K (dQ)
          const CUtensorMap* mb = (role == kRoleAccP) ? &tmA0 : &tmA1;
          for (int n = 0; ok && n < x.N; ++n) {
            const int rows = step_rows<DIR>(g, x, n), hd = step_head<DIR>(g, x, n);
            for (int c = 0; c < DH / 256; ++c, ++issued) {
              const int s = issued % NR_A;
              if (issued >= NR_A && !mbar_wait_cl(&bars->ring_empty[s], ((issued / NR_A) & 1) ^ 1, abort_flag, R)) {
                ok = false;
                break;
              }
              if (leader) mbar_arrive_expect_tx(&bars->ring_full[s], 2 * SLOT_A);
              tma_load_4d_pair(base + OFF_RING_A + s * SLOT_A, mb, mapa(smem_u32(&bars->ring_full[s]), lead), 0,
                               rows, 4 * c + 2 * (int)h, hd);
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
      if (!acc_role) {
        const uint32_t idS = idesc_f16(2 * T, T, 0, 0, 0, 0);  // M = 256 (the pair's rows), both K-major
        const uint64_t yd = smem_desc_sw128(sbase, 16, 1024);  // resident dP operand
        const uint32_t x_tm = tmem + X_COL, s_tm = tmem + S_COL, dp_tm = tmem + DP_COL;
        const uint64_t rd = smem_desc_sw128(sbase + OFF_RING_P, 16, 1024);
        // Own step M takes ring loads 8 M .. 8 M + 7: load k of the step sits
        // in slot k % 4 with phase parity k / 4, both fixed at compile time,
        // so the unrolled issue below is MMAs with constant operand offsets
        // (a single thread issues every MMA of the pair; its per-instruction
        // work bounds the rate at which the tensor pipe is fed).
        static_assert(NR_P == 4 && 2 * (DH / 128) == 8, "slot and parity of load k are k % 4 and k / 4");
        int kp = 0, M = 0;  // items with own steps so far, own steps so far
        for (int k = 0; ok; ++k) {
          const int id = get_item(k, ok);
          if (id < 0) break;
          const Item x = make_item<DIR>(g, id, npairs, LX, h);
          const int n_own = own_steps<NPP>(x.N, pp);
          if (n_own == 0) continue;
          // both CTAs: the item's resident S operand is in Tensor Memory -> tell the leader
          ok = mbar_wait_cl(&bars->x_ready, kp & 1, abort_flag, R);
          if (ok) {
            tc_fence_after();
            tc_fence_before();
            arrive_leader(&bars->pair_ready, leader, lead);
          }
          if (leader && ok)
            ok = mbar_wait_cl(&bars->res_full, kp & 1, abort_flag, R) &&
                 mbar_wait_cl(&bars->pair_ready, kp & 1, abort_flag, R);
          ++kp;
          if (!leader) continue;
          for (int m = 0; ok && m < n_own; ++m, ++M) {
            // S of step M (slices 0-3) once the elementwise warps read S of step M - 1, then dP
            // (slices 4-7) once they read dP of step M - 1: each overlaps the other's readout
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              if ((kk & 3) == 0) {
                if (M >= 1 && !mbar_wait_cl(kk == 0 ? &bars->s_free : &bars->p_free, (M - 1) & 1, abort_flag, R)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
              }
              if (!mbar_wait_cl(&bars->ring_full[kk & 3], (kk >> 2) & 1, abort_flag, R)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t sd = desc_add(rd, (kk & 3) * SLOT_P);
#pragma unroll
              for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                  const int c = 2 * (kk & 3) + cc;  // 64-column chunk of the head dim
                  const uint64_t bdk = desc_add(sd, cc * HT * 128 + ks * 32);
                  if (kk < 4)  // S += X[:, chunk] slice^T, X from Tensor Memory (8 columns per 16 elements)
                    mma_pair_ts(s_tm, x_tm + c * 32 + ks * 8, bdk, idS, (c | ks) ? 1u : 0u);
                  else
                    mma_pair_ss(dp_tm, desc_add(yd, c * T * 128 + ks * 32), bdk, idS, (c | ks) ? 1u : 0u);
                }
              }
              mma_commit_pair(&bars->ring_empty[kk & 3], pmask);
              if (kk == 3) mma_commit_pair(&bars->s_full, pmask);
              if (kk == 7) mma_commit_pair(&bars->p_full, pmask);
            }
          }
        }
      } else if (leader) {
        const uint32_t idA = idesc_f16(2 * T, 256, 0, 0, 0, 1);  // A K-major (fp16 tile), B MN-major
        int used = 0;      // ring loads consumed
        int ka = 0;        // items accumulated so far
        int J0 = 0, J1 = 0, J2 = 0;  // own steps of producer pairs 0, 1, 2 consumed so far
        static_assert(NPP <= 3, "producer pairs");
        for (int k = 0; ok; ++k) {
          const int id = get_item(k, ok);
          if (id < 0) break;
          const Item x = make_item<DIR>(g, id, npairs, LX, h);
          if (x.N == 0) continue;
          // both CTAs' epilogues have read the previous item's accumulator out
          if (ka > 0 && !mbar_wait_cl(&bars->acc_free, (ka - 1) & 1, abort_flag, R)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int n = 0; ok && n < x.N; ++n) {
            // step n comes from producer pair n % NPP, its own step j, into slot (n % NPP) RS + j % RS
            const int pr = n % NPP;
            const int j = (pr == 0 ? J0 : (pr == 1 ? J1 : J2)) + n / NPP, slot = pr * RS + j % RS, ph = (j / RS) & 1;
            if (!mbar_wait_cl(&bars->recv_full[slot][0], ph, abort_flag, R) ||
                !mbar_wait_cl(&bars->recv_full[slot][1], ph, abort_flag, R) ||
                !mbar_wait_cl(&bars->peer_recv[slot], ph, abort_flag, R)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t ad = smem_desc_sw128(sbase + OFF_RECV + slot * TILE_BYTES, 16, 1024);
            for (int c = 0; c < DH / 256; ++c, ++used) {
              const int s = used % NR_A;
              if (!mbar_wait_cl(&bars->ring_full[s], (used / NR_A) & 1, abort_flag, R)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t bd = smem_desc_sw128(sbase + OFF_RING_A + s * SLOT_A, T * 128, 1024);
#pragma unroll
              for (int ks = 0; ks < T / 16; ++ks)
                mma_pair_ss(tmem + c * 256, desc_add(ad, (ks >> 2) * T * 128 + (ks & 3) * 32),
                            desc_add(bd, ks * 2048), idA, (n | ks) ? 1u : 0u);
              mma_commit_pair(&bars->ring_empty[s], pmask);
            }
            if (!ok) break;
            mma_commit_pair(&bars->mma_done[slot], pmask);
          }
          if (!ok) break;
          J0 += own_steps<NPP>(x.N, 0);
          J1 += own_steps<NPP>(x.N, 1);
          if (NPP > 2) J2 += own_steps<NPP>(x.N, 2);
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
    } else if (!acc_role && !leader && elect_one()) {
      // ---------------------------------------------------------- relay (producer peer)
      // the peer's 8 warps arrive locally; one remote arrival per step tells the leader
      bool ok = true;
      int M = 0;
      for (int k = 0; ok; ++k) {
        const int id = get_item(k, ok);
        if (id < 0) break;
        const Item x = make_item<DIR>(g, id, npairs, LX, h);
        const int n_own = own_steps<NPP>(x.N, pp);
        for (int m = 0; m < n_own; ++m, ++M) {
          if (!mbar_wait_cl(&bars->s_free, M & 1, abort_flag, R)) {
            ok = false;
            break;
          }
          mbar_arrive_remote(mapa(smem_u32(&bars->s_free), lead));
          if (!mbar_wait_cl(&bars->p_free, M & 1, abort_flag, R)) {
            ok = false;
            break;
          }
          mbar_arrive_remote(mapa(smem_u32(&bars->p_free), lead));
        }
      }
    }
  } else if (warp == kStoreWarp) {
    // ------------------------------------------------------------ tile stores (producers)
    if (!acc_role && elect_one()) {
      // in the order the warpgroups stage them: per own step P (dK/dV pass)
      // then dS, each as two 16 KB halves into the scratch of the accumulator
      // CTA of this half, which is told once both halves are written
      int sm_dst[2];
      for (int kind = 0; kind < 2; ++kind) {
        const uint32_t dst = (kind == 0 ? kAccP : kAccDS) + h;
        asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(sm_dst[kind]) : "r"(mapa(smem_u32(&bars->smid), dst))
                     : "memory");
      }
      bool ok = (DIR == kDirQ || sm_dst[0] >= 0) && sm_dst[1] >= 0;
      if (!ok) cluster_abort(abort_flag, R);
      int ci = 0;  // tiles staged per warpgroup so far
      int M = 0;   // own steps so far
      for (int k = 0; ok; ++k) {
        const int id = get_item(k, ok);
        if (id < 0) break;
        const Item x = make_item<DIR>(g, id, npairs, LX, h);
        const int n_own = own_steps<NPP>(x.N, pp);
        for (int m = 0; ok && m < n_own; ++m, ++M) {
          const int slot = pp * RS + M % RS;
          for (int kind = (DIR == kDirKV ? 0 : 1); ok && kind < 2; ++kind, ++ci) {
            const uint32_t dst = (kind == 0 ? kAccP : kAccDS) + h;
            if (M >= RS && !mbar_wait_cl(&bars->scratch_free[kind][M % RS], ((M / RS) - 1) & 1, abort_flag, R)) {
              ok = false;
              break;
            }
            fence_proxy_async_global();
            unsigned char* gdst = g_tile_scratch + ((size_t)sm_dst[kind] * kMaxRecv + slot) * TILE_BYTES;
            for (int w = 0; w < 2; ++w) {
              if (!mbar_wait_cl(&bars->staged[w], ci & 1, abort_flag, R)) {
                ok = false;
                break;
              }
              bulk_store_s2g(gdst + w * HALF_BYTES, sbase + OFF_STG + w * HALF_BYTES, HALF_BYTES);
              bulk_commit_group();
            }
            if (!ok) break;
            bulk_wait_read_all();
            mbar_arrive(&bars->stg_free[0]);
            mbar_arrive(&bars->stg_free[1]);
            bulk_wait_all();
            fence_proxy_async_global();
            mbar_arrive_remote(mapa(smem_u32(&bars->tile_ready[slot]), dst));
          }
        }
      }
      bulk_wait_all();  // no store still reads this CTA's shared memory
    }
  } else if (!acc_role) {
    // ------------------------------------------------------------ elementwise (producers, both CTAs)
    const int wg = (warp - 2) >> 2, q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const float sl2 = g.scale * kLog2e;
    const int cb0 = 64 * wg;
    const uint32_t stg = sbase + OFF_STG + wg * HALF_BYTES;
    const uint32_t stg_row = stg + r * 128;
    const bool issuer = (warp & 3) == 2;  // warp 2 / 6 loads its warpgroup's step statistics
    int copies = 0;                       // copies out of this warpgroup's staging half
    bool ok = true;
    // stage one 64-column half tile for the store thread
    auto send = [&](const uint32_t (&o)[32]) -> bool {
      if (copies > 0 && !__all_sync(0xffffffffu, mbar_wait_cl(&bars->stg_free[wg], (copies - 1) & 1, abort_flag, R)))
        return false;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        st_smem_v4(stg_row + ((u ^ (r & 7)) << 4), o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
      fence_proxy_async_smem();
      mbar_arrive(&bars->staged[wg]);
      ++copies;
      return true;
    };
    // dK/dV pass: the statistics of an own step's 64 columns of this
    // warpgroup (lse * log2e, then Delta) are bulk-copied into shared memory
    // while the previous step is finished; every thread then reads them by
    // broadcast
    const uint32_t lse_s = sbase + OFF_STATS + wg * 512, dl_s = lse_s + 256;
    int st_issued = 0;
    auto load_stats = [&](const Item& x, int m) {
      const int n = pp + NPP * m;
      const float* src = p.stats + (size_t)step_head<DIR>(g, x, n) * p.Lpad + step_rows<DIR>(g, x, n) + cb0;
      mbar_arrive_expect_tx(&bars->stats_full[wg], 512);
      bulk_load_g2s(lse_s, src, 256, &bars->stats_full[wg]);
      bulk_load_g2s(dl_s, src + (size_t)g.B * g.Hq * p.Lpad, 256, &bars->stats_full[wg]);
      ++st_issued;
    };
    int M = 0;  // own steps so far
    for (int k = 0; ok; ++k) {
      const int id = get_item_warp(k, ok);
      if (id < 0) break;
      const Item x = make_item<DIR>(g, id, npairs, LX, h);
      const int n_own = own_steps<NPP>(x.N, pp);
      if (n_own == 0) continue;
      const int row = x.r0 + r;  // key (KV) or query (Q) of this thread
      const bool row_ok = row < LX;
      {
        // resident S operand into Tensor Memory: row r, fp16 pairs -> one 32-bit column each;
        // warpgroup wg fills columns [128 wg, 128 wg + 128) (head-dim elements [256 wg, 256 wg + 256)).
        // The previous item's S MMAs, the only readers, finished: their
        // s_full was seen before its last S was read.
        const uint4* src =
            reinterpret_cast<const uint4*>(p.x16 + ((size_t)x.head * LX + (row_ok ? row : 0)) * DH) + wg * 32;
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
        mbar_arrive(&bars->x_ready);
      }
      float2 rs_row = make_float2(0.f, 0.f);
      if (DIR == kDirQ && row_ok)
        rs_row =
            make_float2(p.stats[(size_t)x.head * p.Lpad + row], p.stats[((size_t)g.B * g.Hq + x.head) * p.Lpad + row]);
      if (DIR == kDirKV && issuer && lane == 0) {
        // the warpgroup has read the previous step's statistics
        if (M > 0 && !mbar_wait_cl(&bars->stats_free[wg], (M - 1) & 1, abort_flag, R)) ok = false;
        else load_stats(x, 0);
      }
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      for (int m = 0; m < n_own; ++m, ++M) {
        const int n = pp + NPP * m;
        const int c0 = step_rows<DIR>(g, x, n);  // first column's query (KV) or key (Q)
        if (!__all_sync(0xffffffffu, mbar_wait_cl(&bars->s_full, M & 1, abort_flag, R))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sv[64], dv[64];
        tmem_ld32(tmem + lane_off + S_COL + cb0, *reinterpret_cast<uint32_t(*)[32]>(sv));
        tmem_ld32(tmem + lane_off + S_COL + cb0 + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_free);  // S may be overwritten (the peer's relay tells the leader)
        bool full;
        int4 vv;
        if (DIR == kDirKV) {  // columns are query rows c0 .. c0 + 127, this thread's row is key `row`
          full = x.own_rows && keys_tile_full(g, x.r0, x.rlast, c0, c0 + T - 1);
          vv = key_vis(g, row, c0);
        } else {  // columns are keys c0 .. c0 + 127, this thread's row is query `row`
          full = x.own_rows && rows_tile_full(g, x.r0, x.rlast, c0, c0 + T - 1);
          vv = row_vis(g, row, c0);
        }
        if (DIR == kDirKV && !__all_sync(0xffffffffu, mbar_wait_cl(&bars->stats_full[wg], M & 1, abort_flag, R))) {
          ok = false;
          break;
        }
        bool both;
        vv = vis_in_tile(vv, T, &both);
        const bool two_here = two && __any_sync(0xffffffffu, both);
        if (full) p_tile64<true, DIR == kDirKV>(sv, lse_s, rs_row.x, sl2, cb0, vv);
        else if (two_here) p_tile64<false, DIR == kDirKV, true>(sv, lse_s, rs_row.x, sl2, cb0, vv);
        else p_tile64<false, DIR == kDirKV>(sv, lse_s, rs_row.x, sl2, cb0, vv);
        uint32_t o[32];
        if (DIR == kDirKV) {
          pack64(sv, o);
          if (!send(o)) {  // P^T -> dV accumulator
            ok = false;
            break;
          }
        }
        if (!__all_sync(0xffffffffu, mbar_wait_cl(&bars->p_full, M & 1, abort_flag, R))) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_ld32(tmem + lane_off + DP_COL + cb0, *reinterpret_cast<uint32_t(*)[32]>(dv));
        tmem_ld32(tmem + lane_off + DP_COL + cb0 + 32, *reinterpret_cast<uint32_t(*)[32]>(dv + 32));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_free);  // dP may be overwritten
        ds_tile64<DIR == kDirKV>(sv, dv, dl_s, rs_row.y, o);
        if (DIR == kDirKV) {
          // the warpgroup has read this step's statistics: the next step's may land
          mbar_arrive(&bars->stats_free[wg]);
          if (issuer && lane == 0 && m + 1 < n_own) {
            if (!mbar_wait_cl(&bars->stats_free[wg], M & 1, abort_flag, R)) ok = false;
            else load_stats(x, m + 1);
          }
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
        }
        if (!send(o)) {  // dS -> dK / dQ accumulator
          ok = false;
          break;
        }
      }
    }
    // unwinding: the last statistics load must have landed (the store thread
    // waits for its own stores)
    if (st_issued > 0) mbar_wait_drain(&bars->stats_full[wg], (st_issued - 1) & 1);
  } else {
    // ------------------------------------------------------------ accumulator warps 2-9 (both CTAs)
    const int wg = (warp - 2) >> 2, q4 = warp & 3;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const float inv_s = p.stats[dscale_offset(g, p.Lpad) + 1];  // 1/s of the scaled dO copy
    const float mul = (DIR == kDirKV && role == kRoleAccP) ? inv_s : g.scale * inv_s;
    float* const out = (DIR == kDirKV && role == kRoleAccP) ? p.out1 : p.out0;
    const CUtensorMap* om = (DIR == kDirKV && role == kRoleAccP) ? &tmO1 : &tmO0;
    const bool loader = warp >= 2 + NPP && warp < 2 + 2 * NPP;  // one per producer pair
    const bool watcher = warp >= 2 && warp < 2 + NPP;           // one per producer pair
    const int p2 = loader ? warp - 2 - NPP : warp - 2;          // the pair a loader or watcher serves
    const unsigned char* scr = g_tile_scratch + (size_t)(bars->smid < 0 ? 0 : bars->smid) * kMaxRecv * TILE_BYTES;
    bool ok = true;
    if (loader && bars->smid < 0) {
      ok = false;
      if (lane == 0) cluster_abort(abort_flag, R);
    }
    int J = 0;   // own steps of pair p2 handled so far (loaders and watchers)
    int ka = 0;  // items accumulated so far
    for (int k = 0; ok; ++k) {
      const int id = get_item_warp(k, ok);
      if (id < 0) break;
      const Item x = make_item<DIR>(g, id, npairs, LX, h);
      if (x.N == 0) {
        // dK/dV pass, and no query sees these keys (queries that are a suffix
        // of the keys, with a window): zero gradients ("Lab 028 lab detail",
        // "What I changed, in plain terms" item 5(b))
        zero_rows(out, x.head, x.r0, T, g.L, DH, (int)threadIdx.x - 64, 256);
        continue;
      }
      const int nown = (loader || watcher) ? own_steps<NPP>(x.N, p2) : 0;
      if (loader && lane == 0) {
        // once the MMAs are done with a slot and the producer's tile is in
        // the scratch, load it into the slot; the receive slots held the
        // previous item's epilogue staging until its stores had read it
        if (ka > 0 && !mbar_wait_cl(&bars->epi_done, (ka - 1) & 1, abort_flag, R)) ok = false;
        for (int j = J; ok && j < J + nown; ++j) {
          const int slot = p2 * RS + j % RS, ph = (j / RS) & 1;
          if (j >= RS && !mbar_wait_cl(&bars->mma_done[slot], ((j / RS) - 1) & 1, abort_flag, R)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->recv_full[slot][0], HALF_BYTES);
          mbar_arrive_expect_tx(&bars->recv_full[slot][1], HALF_BYTES);
          if (!mbar_wait_cl(&bars->tile_ready[slot], ph, abort_flag, R)) {
            // armed but never loaded: the drain below does not wait on it
            ok = false;
            break;
          }
          fence_proxy_async_global();
          bulk_load_g2s(sbase + OFF_RECV + slot * TILE_BYTES, scr + (size_t)slot * TILE_BYTES, HALF_BYTES,
                        &bars->recv_full[slot][0]);
          bulk_load_g2s(sbase + OFF_RECV + slot * TILE_BYTES + HALF_BYTES,
                        scr + (size_t)slot * TILE_BYTES + HALF_BYTES, HALF_BYTES, &bars->recv_full[slot][1]);
          bars->n_loaded[p2] = j + 1;
        }
      }
      if (watcher && lane == 0) {
        // when both halves of a tile are in the slot, the producer may reuse
        // that scratch slot; the peer also tells the leader that its rows of
        // the step's A operand are here
        const uint32_t prod = (uint32_t)(2 * p2) + h;
        for (int j = J; j < J + nown; ++j) {
          const int slot = p2 * RS + j % RS, ph = (j / RS) & 1;
          if (!mbar_wait_cl(&bars->recv_full[slot][0], ph, abort_flag, R) ||
              !mbar_wait_cl(&bars->recv_full[slot][1], ph, abort_flag, R)) {
            ok = false;
            break;
          }
          bars->n_recv[p2] = j + 1;
          mbar_arrive_remote(mapa(smem_u32(&bars->scratch_free[dst_kind][j % RS]), prod));
          if (!leader) mbar_arrive_remote(mapa(smem_u32(&bars->peer_recv[slot]), lead));
        }
      }
      J += nown;
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      if (!__all_sync(0xffffffffu, mbar_wait_cl(&bars->acc_done, ka & 1, abort_flag, R))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // every receive slot has been consumed by the finished MMAs: each of
      // warps 2-9 stages its blocks in NRECV 4 KB buffers there (an eighth
      // of the slots; the ring after them may already hold the next item's
      // loads)
      static_assert(8 * NRECV * 4096 == NRECV * TILE_BYTES && NRECV <= 4, "epilogue staging fills the receive slots");
      tmem_rows_store_tma<NRECV, false>(om, tmem + lane_off + 256 * wg, 256 * wg, 256, mul,
                                        sbase + OFF_RECV + (uint32_t)(warp - 2) * (NRECV * 4096u), x.r0 + 32 * q4,
                                        x.head, lane);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars->epi_done);                   // the staging may be overwritten
        arrive_leader(&bars->acc_free, leader, lead);  // the accumulator may be overwritten
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
    // unwinding only.  Accumulators: tile loads issued but never observed
    // must land before this CTA's shared memory is released.
    if (acc_role) {
      // (the last load into each slot: earlier ones on the same barrier
      // completed before it)
      for (int pr = 0; pr < NPP; ++pr)
        for (int j = max(bars->n_recv[pr], bars->n_loaded[pr] - RS); j < bars->n_loaded[pr]; ++j) {
          mbar_wait_drain(&bars->recv_full[pr * RS + j % RS][0], (j / RS) & 1);
          mbar_wait_drain(&bars->recv_full[pr * RS + j % RS][1], (j / RS) & 1);
        }
    }
    // Leader: the ring and resident loads of both CTAs complete on its
    // barriers; let the last load of each slot (of either CTA) land.
    if (leader) {
      int peer_issued, peer_res;
      asm volatile("ld.shared::cluster.u32 %0, [%1];"
                   : "=r"(peer_issued)
                   : "r"(mapa(smem_u32(&bars->n_issued), lead + 1))
                   : "memory");
      asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(peer_res) : "r"(mapa(smem_u32(&bars->n_res), lead + 1))
                   : "memory");
      const int issued = max(bars->n_issued, peer_issued);
      const int nr = acc_role ? NR_A : NR_P;
      for (int k = issued - 1; k >= 0 && k >= issued - nr; --k)
        mbar_wait_drain(&bars->ring_full[k % nr], (k / nr) & 1);
      const int n_res = max(bars->n_res, peer_res);
      if (!acc_role && n_res > 0) mbar_wait_drain(&bars->res_full, (n_res - 1) & 1);
    }
  }
  __syncthreads();
  cluster_sync();
  if (*abort_flag && threadIdx.x == 0) atomicCAS(p.status, 0, kStatusTimeout);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
  // dQ pass started early beside the dK/dV pass: it completes after that
  // pass, so that whatever follows on the stream sees both finished
  if (DIR == kDirQ && threadIdx.x == 0) grid_dependency_wait();
}

// Clusters of a pass that fit on the current device at once (cached per
// device; 0 on an error).
template <int DIR>
int max_clusters(const cudaLaunchConfig_t& cfg) {
  static std::atomic<int> cached[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < kMaxDevices) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, bwd512_kernel<DIR>, &cfg) != cudaSuccess) return 0;
  if (dev < kMaxDevices && n > 0) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <int DIR>
cudaError_t launch_pair(const Geom& g, const uint16_t* q16, const uint16_t* k16, const uint16_t* v16,
                        const uint16_t* g16, const float* stats, int Lpad, float* out0, float* out1, int* status,
                        cudaStream_t s, bool early) {
  // streamed operands (64-row halves, two chunks per slice), the resident dP
  // operand (one chunk of 128 rows per load), accumulator operands (two chunks
  // of 128 rows per load)
  CUtensorMap tmS, tmP, tmR, tmA0, tmA1, tmO0, tmO1;
  cudaError_t e;
  // fp32 outputs: [B Hkv, L, D] dk and dv (dK/dV pass), [B Hq, Lq, D] dq (dQ pass)
  if (DIR == kDirKV) {
    if ((e = make_tmap_f32_out(&tmO0, out0, DH, g.L, g.B * g.Hkv)) != cudaSuccess) return e;
    if ((e = make_tmap_f32_out(&tmO1, out1, DH, g.L, g.B * g.Hkv)) != cudaSuccess) return e;
  } else {
    if ((e = make_tmap_f32_out(&tmO0, out0, DH, g.Lq, g.B * g.Hq)) != cudaSuccess) return e;
    tmO1 = tmO0;
  }
  if (DIR == kDirKV) {
    if ((e = make_tmap_f16_chunks(&tmS, q16, DH, g.Lq, g.B * g.Hq, HT, 2)) != cudaSuccess) return e;
    if ((e = make_tmap_f16_chunks(&tmP, g16, DH, g.Lq, g.B * g.Hq, HT, 2)) != cudaSuccess) return e;
    if ((e = make_tmap_f16(&tmR, v16, DH, g.L, g.B * g.Hkv, T)) != cudaSuccess) return e;
    if ((e = make_tmap_f16_chunks(&tmA0, g16, DH, g.Lq, g.B * g.Hq, T, 2)) != cudaSuccess) return e;
    if ((e = make_tmap_f16_chunks(&tmA1, q16, DH, g.Lq, g.B * g.Hq, T, 2)) != cudaSuccess) return e;
  } else {
    if ((e = make_tmap_f16_chunks(&tmS, k16, DH, g.L, g.B * g.Hkv, HT, 2)) != cudaSuccess) return e;
    if ((e = make_tmap_f16_chunks(&tmP, v16, DH, g.L, g.B * g.Hkv, HT, 2)) != cudaSuccess) return e;
    if ((e = make_tmap_f16(&tmR, g16, DH, g.Lq, g.B * g.Hq, T)) != cudaSuccess) return e;
    if ((e = make_tmap_f16_chunks(&tmA0, k16, DH, g.L, g.B * g.Hkv, T, 2)) != cudaSuccess) return e;
    if ((e = make_tmap_f16_chunks(&tmA1, k16, DH, g.L, g.B * g.Hkv, T, 2)) != cudaSuccess) return e;
  }
  auto kern = bwd512_kernel<DIR>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM)) != cudaSuccess)
    return e;
  ParamsPair pm;
  pm.g = g;
  // the pass's work counter in the stats tail, zeroed by the absmax pass
  pm.work = reinterpret_cast<int*>(const_cast<float*>(stats) + dscale_offset(g, Lpad) + kWorkCounterFloat + DIR);
  pm.out0 = out0;
  pm.out1 = out1;
  pm.x16 = (DIR == kDirKV) ? k16 : q16;
  pm.stats = stats;
  pm.Lpad = Lpad;
  pm.n_tiles = ((DIR == kDirKV ? g.L : g.Lq) + T - 1) / T;  // resident-side tiles
  pm.n_items = g.B * g.Hkv * ((pm.n_tiles + 1) / 2) * (DIR == kDirQ ? g.G : 1);
  pm.status = status;
  constexpr unsigned R = PassCfg<DIR>::R;
  if (R > 8 && (e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(R, 1, 1);
  cfg.blockDim = dim3(kThr, 1, 1);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = R;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // persistent clusters: as many as fit on the GPU at once, at most one per item
  const int fit = max_clusters<DIR>(cfg);
  if (fit <= 0) return cudaErrorInvalidConfiguration;
  cfg.gridDim = dim3(R * (unsigned)min(fit, pm.n_items), 1, 1);
  if (early) cfg.numAttrs = 2;  // may start before the kernel ahead of it on `s` has finished
  return cudaLaunchKernelEx(&cfg, kern, tmS, tmP, tmR, tmA0, tmA1, tmO0, tmO1, pm);
}

}  // namespace

int scratch_layout_bwd512() {
  int n0 = 0, n1 = 0, nsm = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev))
    return -1;
  if (cudaFuncSetAttribute(bwd512_kernel<kDirKV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM) ||
      cudaFuncSetAttribute(bwd512_kernel<kDirQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM) ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n0, bwd512_kernel<kDirKV>, kThr, SMEM) ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n1, bwd512_kernel<kDirQ>, kThr, SMEM))
    return -1;
  return (n0 == 1 && n1 == 1 && nsm <= kScratchSms) ? 0 : 1;
}

cudaError_t launch_bwd_dkdv_tc512(const Geom& g, const uint16_t* q16, const uint16_t* k16, const uint16_t* v16,
                                   const uint16_t* g16, const float* stats, int Lpad, float* dk, float* dv,
                                   int* status, cudaStream_t s) {
  return launch_pair<kDirKV>(g, q16, k16, v16, g16, stats, Lpad, dk, dv, status, s, false);
}

cudaError_t launch_bwd_dq_tc512(const Geom& g, const uint16_t* q16, const uint16_t* k16, const uint16_t* v16,
                                 const uint16_t* g16, const float* stats, int Lpad, float* dq, int* status,
                                 cudaStream_t s) {
  return launch_pair<kDirQ>(g, q16, k16, v16, g16, stats, Lpad, dq, nullptr, status, s, true);
}

}  // namespace swa
