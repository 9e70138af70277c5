// Dynamic claiming of work items by the persistent CTAs of the three
// attention kernels.
//
// Each work list is ordered longest first (geometry.cuh).  The CTAs take its
// items in that order as they become free: one thread per CTA (the producer)
// claims the next index from a counter in global memory and hands it to the
// CTA's other roles through a ring of kRingSlots slots in shared memory, one
// round (item) per slot.  A CTA that runs slower -- its SM is slower, or its
// items ran longer -- claims fewer items, so the grid finishes together; a
// static assignment of equal work per CTA ends with its slowest SM.  The items
// running at any moment stay a window of about one grid's worth of
// consecutive list items, which keeps the list's KV-head blocking intact.
//
// The counter and a count of finished CTAs are two words of the workspace
// header, zeroed before every call; the last CTA to finish zeroes them again,
// so one call may launch a kernel more than once.  The load-balancing
// ablation (Geom::naive_order) keeps the static round-robin assignment
// (round r of CTA c: item r * grid + c) through the same ring.
#pragma once
#include "geometry.cuh"
#include "ptx.cuh"

namespace bdlm {

constexpr int kRingSlots = 4;

struct ItemRing {
  uint32_t full;              // shared address of kRingSlots barriers (1 arrival: the producer)
  uint32_t empty;             // kRingSlots barriers (one arrival per consumer thread)
  volatile int64_t* slot;     // kRingSlots item indices
};

// Shared-memory footprint of a ring: 2 * kRingSlots barriers + kRingSlots slots.
constexpr int kRingBytes = 2 * kRingSlots * 8 + kRingSlots * 8;

// Producer: the index of its CTA's round `rnd` item.
__device__ __forceinline__ int64_t claim_item(const Geom& g, uint32_t* counter, int64_t rnd, int cta, int grid) {
  return g.naive_order ? rnd * grid + cta : (int64_t)atomicAdd(counter, 1u);
}

// Producer, in two parts for rings whose slots carry more than the index
// (the caller writes its own part of slot rnd % kRingSlots in between):
// waits for round rnd's slot to be free ...
__device__ __forceinline__ bool ring_acquire(const ItemRing& r, int64_t rnd, const Watchdog& wd, uint32_t site) {
  const uint32_t s = (uint32_t)rnd & (kRingSlots - 1);
  const uint32_t use = (uint32_t)(rnd / kRingSlots);
  return use == 0 || mbar_wait(r.empty + 8 * s, (use - 1) & 1, wd, site);
}
// ... and publishes round rnd's item.
__device__ __forceinline__ void ring_publish(const ItemRing& r, int64_t rnd, int64_t idx) {
  const uint32_t s = (uint32_t)rnd & (kRingSlots - 1);
  r.slot[s] = idx;
  mbar_arrive(r.full + 8 * s);
}

// Producer: publishes round rnd's item (waits for its slot to be free).
__device__ __forceinline__ bool ring_put(const ItemRing& r, int64_t rnd, int64_t idx, const Watchdog& wd,
                                         uint32_t site) {
  if (!ring_acquire(r, rnd, wd, site)) return false;
  ring_publish(r, rnd, idx);
  return true;
}

// Consumer thread, in two parts: waits for round rnd's item ...  (Every
// consumer thread arrives on its own, with no warp-wide step, so that a
// thread that gives up after a wait limit never leaves its warp's other
// lanes waiting for it.)
__device__ __forceinline__ bool ring_wait(const ItemRing& r, int64_t rnd, int64_t& idx, const Watchdog& wd,
                                          uint32_t site) {
  const uint32_t s = (uint32_t)rnd & (kRingSlots - 1);
  if (!mbar_wait(r.full + 8 * s, (uint32_t)(rnd / kRingSlots) & 1, wd, site)) return false;
  idx = r.slot[s];
  return true;
}
// ... and, once it no longer reads the slot, frees it.
__device__ __forceinline__ void ring_release(const ItemRing& r, int64_t rnd) {
  mbar_arrive(r.empty + 8 * ((uint32_t)rnd & (kRingSlots - 1)));
}

// Consumer thread: round rnd's item, its slot freed at once.
__device__ __forceinline__ bool ring_get(const ItemRing& r, int64_t rnd, int64_t& idx, const Watchdog& wd,
                                         uint32_t site) {
  if (!ring_wait(r, rnd, idx, wd, site)) return false;
  ring_release(r, rnd);
  return true;
}

// One thread per CTA, after the CTA's last claim: the last CTA of the grid
// to get here zeroes the counter and the finished count for the next launch.
__device__ __forceinline__ void sched_release(uint32_t* counter, int grid) {
  __threadfence();
  if (atomicAdd(counter + 1, 1u) == (uint32_t)grid - 1) {
    atomicExch(counter, 0u);
    atomicExch(counter + 1, 0u);
    __threadfence();
  }
}

}  // namespace bdlm
