// Work items of a persistent thread-block cluster (the head-dim-512 kernels).
//
// A persistent launch has as many clusters as fit on the GPU at once; each
// cluster loops over work items, whose ids it draws from a counter in global
// memory that is zero when the launch starts.  Rank 0 of the cluster runs the
// scheduler in one thread of an otherwise idle warp:
//   - it draws an id (atomicAdd; -1 once the ids run out) and writes it into
//     slot k % 2 of every CTA of the cluster (remote st.shared::cluster), then
//     fence.acq_rel.cluster and one relaxed remote arrive on each CTA's
//     full[k % 2] barrier, so the id is visible before the arrive is seen;
//   - it reuses a slot only once every reader of its previous id has reported
//     on rank 0's empty[] barrier;
//   - it draws id k only after rank 0's TMA thread has requested it (req),
//     which that thread does when it starts the last step of its current
//     item.  Clusters then take items in about the order they finish them,
//     as the clusters of a non-persistent grid would be dispatched, and the
//     clusters of one kv head walk its tiles about in step, sharing them in
//     L2 (drawing as soon as a slot is free tripled one pass's DRAM reads).
// Every wait is bounded and gives up when the cluster's abort flag is raised.
#pragma once

#include <stdint.h>

#include "tc_ptx.cuh"

namespace swa {
namespace tc {

struct ItemRing {
  uint64_t full[2];   // (every CTA) the scheduler wrote an item id into the slot
  uint64_t empty[2];  // (rank 0) every reader of the slot read it
  uint64_t req;       // (rank 0) its TMA thread will soon need the next item
  int id[2];          // item ids, written by rank 0's scheduler
};

// One thread of every CTA, before the cluster barrier that precedes any use.
// readers: the arrivals the scheduler waits for on each slot (every thread or
// warp that reads ids reports once per id, across the whole cluster).
__device__ __forceinline__ void item_ring_init(ItemRing* r, int readers) {
  for (int s = 0; s < 2; ++s) {
    mbar_init(&r->full[s], 1);
    mbar_init(&r->empty[s], readers);
  }
  mbar_init(&r->req, 1);
}

// The k-th item of this cluster (k = 0, 1, ...): its id, or -1 once the work
// has run out or after a timeout (then ok is cleared).  One thread.
__device__ __forceinline__ int item_get(ItemRing* r, int k, bool& ok, volatile int* abort, uint32_t nranks) {
  if (!mbar_wait_cl(&r->full[k & 1], (k >> 1) & 1, abort, nranks)) {
    ok = false;
    return -1;
  }
  const int id = *reinterpret_cast<volatile int*>(&r->id[k & 1]);
  // the id has been used (compared) before the report, so its load is complete
  if (id >= 0) mbar_arrive_remote(mapa(smem_u32(&r->empty[k & 1]), 0));
  return id;
}

// The same for a whole warp; lane 0 reports the read.
__device__ __forceinline__ int item_get_warp(ItemRing* r, int k, bool& ok, volatile int* abort, uint32_t nranks,
                                             int lane) {
  if (!__all_sync(0xffffffffu, mbar_wait_cl(&r->full[k & 1], (k >> 1) & 1, abort, nranks))) {
    ok = false;
    return -1;
  }
  const int id = *reinterpret_cast<volatile int*>(&r->id[k & 1]);
  __syncwarp();
  if (lane == 0 && id >= 0) mbar_arrive_remote(mapa(smem_u32(&r->empty[k & 1]), 0));
  return id;
}

// Rank 0's TMA thread: the next item will soon be needed (once per item).
__device__ __forceinline__ void item_request(ItemRing* r) { mbar_arrive(&r->req); }

// The scheduler (rank 0, one thread): runs until it has published -1 or the
// cluster aborts.
__device__ __forceinline__ void item_schedule(ItemRing* r, int* work, int n_items, volatile int* abort,
                                              uint32_t nranks) {
  for (int k = 0;; ++k) {
    const int s = k & 1;
    if (k >= 1 && !mbar_wait_cl(&r->req, (k - 1) & 1, abort, nranks)) return;
    if (k >= 2 && !mbar_wait_cl(&r->empty[s], ((k >> 1) - 1) & 1, abort, nranks)) return;
    int id = atomicAdd(work, 1);
    if (id >= n_items) id = -1;
    const uint32_t slot_addr = smem_u32(&r->id[s]);
    for (uint32_t c = 0; c < nranks; ++c) st_cluster_u32(mapa(slot_addr, c), (uint32_t)id);
    fence_acq_rel_cluster();  // the ids are visible before any CTA sees the arrive
    for (uint32_t c = 0; c < nranks; ++c) mbar_arrive_remote(mapa(smem_u32(&r->full[s]), c));
    if (id < 0) return;
  }
}

}  // namespace tc
}  // namespace swa
