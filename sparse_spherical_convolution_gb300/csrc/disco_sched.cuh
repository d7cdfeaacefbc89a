// disco_sched.cuh -- dynamic tile scheduling for the persistent kernels.
//
// A persistent kernel (one CTA per SM) takes its next tile from a counter in
// global memory instead of a fixed round-robin share.  Tiles of the DISCO
// contractions differ a lot in cost (near the poles a row's longitude window
// spans many more columns), so a fixed share lets the CTAs drift apart: the
// tiles in flight then spread over many row groups and the L2 no longer
// serves the operand rows that neighbouring groups share.  Taken in order
// from one counter, the tiles in flight stay a contiguous window of the tile
// order.
//
// The counter must be private to one launch, also when several launches run
// at once on different streams, and the library allocates no memory.  So
// each kernel family owns a file-scope table of slots; a launch carries a
// process-unique id (next_launch_id) and uses slot id % kSchedSlots:
//   claim    one thread per CTA swaps the slot's owner from 0 to the id (or
//            finds the id already there, set by a sibling CTA); a slot still
//            held by an earlier launch is waited for, with a bound;
//   next     atomicAdd on the slot's counter;
//   release  the CTA that finishes last resets the counters and frees the
//            slot.
// A claim that times out reports failure: the CTA then takes no tile.
#pragma once

#include <stdint.h>

namespace disco {

constexpr int kSchedSlots = 1024;

struct SchedSlot {
  unsigned long long owner;  // launch id holding the slot, 0 = free
  int next;                  // next tile to hand out
  int done;                  // CTAs of the owner that finished
};

__device__ __forceinline__ SchedSlot* sched_claim(SchedSlot* table, unsigned long long id, uint32_t limit) {
  SchedSlot* s = table + (id % kSchedSlots);
  for (uint32_t i = 0; i < limit; ++i) {
    const unsigned long long o = atomicCAS(&s->owner, 0ull, id);
    if (o == 0ull || o == id) {
      __threadfence();
      return s;
    }
    __nanosleep(200);
  }
  return nullptr;
}

__device__ __forceinline__ int sched_next(SchedSlot* s) { return atomicAdd(&s->next, 1); }

// Called once per CTA that claimed the slot, after its last sched_next.
__device__ __forceinline__ void sched_release(SchedSlot* s) {
  __threadfence();
  if (atomicAdd(&s->done, 1) == (int)(gridDim.x * gridDim.y * gridDim.z) - 1) {
    atomicExch(&s->next, 0);
    atomicExch(&s->done, 0);
    __threadfence();
    atomicExch(&s->owner, 0ull);
  }
}

}  // namespace disco
