// Run-time work distribution for the persistent kernels.
//
// Work items (a q-tile or a k-tile with its heads) are numbered in the plan's
// order and handed out at run time: the producer warp of each CTA takes the
// next number from a global counter, so a CTA that drew short items takes more
// of them and all CTAs finish together (a fixed round-robin split leaves the
// CTAs that drew the long items of a trie's shared prefix running alone).
// The producer passes each number to the CTA's other roles through a ring of
// shared-memory entries guarded by mbarriers; it stays one item ahead, so the
// consumers can look at the next item before they finish the current one.
//
// Counters: each launch takes its own slot of a ring of kSchedSlots counters
// (library-owned device memory) and the last CTA to finish puts it back to
// zero, so launches in flight at the same time on different streams never
// share a counter.
#pragma once

#include "sm103_ptx.cuh"

namespace treeattn {

struct SchedSlot {
  unsigned int next;  // next item number to hand out
  unsigned int done;  // CTAs of the launch that have finished
};

constexpr int kSchedSlots = 1024;

namespace dev {

constexpr uint32_t kItemRing = 8;

struct ItemRing {
  int id[kItemRing];
  int info[kItemRing][3];     // the item's header as the producer decoded it
  uint64_t full[kItemRing];   // one arrival: the producer wrote the entry
  uint64_t empty[kItemRing];  // one arrival per consumer warp: every consumer read it
};

__device__ __forceinline__ void item_ring_init(ItemRing* r, uint32_t consumer_warps) {
  for (uint32_t e = 0; e < kItemRing; ++e) {
    mbar_init(&r->full[e], 1);
    mbar_init(&r->empty[e], consumer_warps);
  }
}

// Producer warp (warp-collective): the next item number, or -1 when the
// launch has none left.
__device__ __forceinline__ int item_fetch(SchedSlot* s, int n_items) {
  int v = 0;
  if ((threadIdx.x & 31) == 0) v = static_cast<int>(atomicAdd(&s->next, 1u));
  v = __shfl_sync(0xffffffffu, v, 0);
  return v < n_items ? v : -1;
}

// Producer warp (warp-collective): publish this CTA's n-th item number and
// (optionally) three ints of its decoded header.
__device__ __forceinline__ bool item_put(ItemRing* r, uint32_t& n, int id, volatile int* abort,
                                         int* status, int a = 0, int b = 0, int c = 0) {
  const uint32_t e = n % kItemRing, ph = (n / kItemRing) & 1;
  bool ok = true;
  if (n >= kItemRing) ok = mbar_wait(&r->empty[e], ph ^ 1, abort, status, kSiteRing + static_cast<int>(threadIdx.x / 32));
  if (!__all_sync(0xffffffffu, ok)) return false;
  if ((threadIdx.x & 31) == 0) {
    reinterpret_cast<volatile int*>(r->id)[e] = id;
    reinterpret_cast<volatile int*>(r->info[e])[0] = a;
    reinterpret_cast<volatile int*>(r->info[e])[1] = b;
    reinterpret_cast<volatile int*>(r->info[e])[2] = c;
    mbar_arrive(&r->full[e]);  // release: the entry is visible to whoever sees the phase flip
  }
  __syncwarp();
  ++n;
  return true;
}

// Consumer warp (warp-collective): this CTA's n-th item number; the entry is
// released as soon as it is read.
__device__ __forceinline__ bool item_get(ItemRing* r, uint32_t& n, int& id, volatile int* abort,
                                         int* status, int* info = nullptr) {
  const uint32_t e = n % kItemRing, ph = (n / kItemRing) & 1;
  const bool ok = mbar_wait(&r->full[e], ph, abort, status, kSiteRing + static_cast<int>(threadIdx.x / 32));
  if (!__all_sync(0xffffffffu, ok)) return false;
  id = reinterpret_cast<volatile int*>(r->id)[e];
  if (info) {
    info[0] = reinterpret_cast<volatile int*>(r->info[e])[0];
    info[1] = reinterpret_cast<volatile int*>(r->info[e])[1];
    info[2] = reinterpret_cast<volatile int*>(r->info[e])[2];
  }
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&r->empty[e]);
  ++n;
  return true;
}

// One thread per CTA, after the CTA's last __syncthreads: the last CTA of the
// launch to get here zeroes the slot for the launch that takes it next. Every
// CTA stops fetching before it gets here, so no fetch can follow the reset.
__device__ __forceinline__ void sched_finish(SchedSlot* s) {
  __threadfence();
  if (atomicAdd(&s->done, 1u) == gridDim.x - 1) {
    reinterpret_cast<volatile unsigned int*>(&s->next)[0] = 0u;
    reinterpret_cast<volatile unsigned int*>(&s->done)[0] = 0u;
    __threadfence();
  }
}

}  // namespace dev
}  // namespace treeattn
