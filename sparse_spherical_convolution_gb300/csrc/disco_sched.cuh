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
// each kernel family owns a file-scope table of 64-bit words; a launch
// carries a process-unique id (next_launch_id) and uses word id % kSchedSlots:
//
//   bits 63..34  tag: the low 30 bits of the id of the launch using the word
//   bits 33..24  active: CTAs of that launch that joined and have not left
//   bits 23..0   next tile to hand out
//
//   join   (once per CTA, compare-and-swap) if the tag is the launch's own,
//          active + 1; if another launch's tag is there with no active CTA,
//          take the word: own tag, active 1, counter 0; otherwise another
//          launch is still drawing: wait, bounded, and give up (the CTA then
//          takes no tile and flags its status bit);
//   next   atomicAdd of 1 (only between a CTA's join and its leave);
//   leave  (once per joined CTA, on every exit path) active - 1.
//
// Only joined CTAs count in `active` and every joined CTA leaves, so once
// all CTAs of a launch have exited its word has no active CTA and the next
// launch that maps to it takes it over: no failure leaves a word held.
// While a CTA draws, its launch's active count is non-zero, so no other
// launch can take the word: every draw lands on the drawing launch's own
// counter.  A CTA that gives up waiting loses no tile (its siblings draw
// them all); a CTA that joins late, after its launch's word was taken over
// and freed, takes it back and recomputes its launch's tiles, whose outputs
// are plain stores of values that depend on the inputs alone.
#pragma once

#include <stdint.h>

namespace disco {

constexpr int kSchedSlots = 1024;
constexpr unsigned long long kSchedCountMask = (1ull << 24) - 1;
constexpr unsigned long long kSchedActiveOne = 1ull << 24;
constexpr unsigned long long kSchedActiveMask = ((1ull << 10) - 1) << 24;
constexpr unsigned long long kSchedTagMask = ~(kSchedCountMask | kSchedActiveMask);
constexpr int kSchedMaxCtas = (1 << 10) - 1;  // CTAs of one launch (active field)

__host__ __device__ __forceinline__ unsigned long long sched_tag(unsigned long long id) {
  return (id & ((1ull << 30) - 1)) << 34;
}

// Joins the launch's word; nullptr if another launch kept drawing from it for
// `limit` polls.  One thread per CTA.
__device__ __forceinline__ unsigned long long* sched_join(unsigned long long* table, unsigned long long id,
                                                          uint32_t limit) {
  unsigned long long* w = table + (id % kSchedSlots);
  const unsigned long long tag = sched_tag(id);
  unsigned long long old = *(volatile unsigned long long*)w;
  for (uint32_t i = 0; i < limit; ++i) {
    unsigned long long want;
    if ((old & kSchedTagMask) == tag) {
      want = old + kSchedActiveOne;
    } else if ((old & kSchedActiveMask) == 0) {
      want = tag | kSchedActiveOne;
    } else {
      __nanosleep(200);
      old = *(volatile unsigned long long*)w;
      continue;
    }
    const unsigned long long seen = atomicCAS(w, old, want);
    if (seen == old) {
      __threadfence();
      return w;
    }
    old = seen;
  }
  return nullptr;
}

// Next tile of the launch (values past its tile count: none left).  The
// launch keeps tiles + CTAs below 2^24 (checked on the host).
__device__ __forceinline__ int sched_next(unsigned long long* w) {
  return (int)(atomicAdd(w, 1ull) & kSchedCountMask);
}

// Once per joined CTA, after its last sched_next.
__device__ __forceinline__ void sched_leave(unsigned long long* w) {
  __threadfence();
  atomicAdd(w, 0ull - kSchedActiveOne);
}

}  // namespace disco
