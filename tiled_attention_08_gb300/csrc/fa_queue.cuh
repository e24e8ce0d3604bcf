// fa_queue.cuh -- dynamic distribution of work items to persistent CTAs (backward passes).
//
// Every persistent CTA takes its next work id from a counter in global memory (atomicAdd),
// so the items, ordered heaviest first, go to whichever CTA frees up first: the greedy
// longest-first schedule, which stays balanced for rows of any length (fixed snake rounds
// balance causal items well only when each CTA takes many small ones).  The counter lives in
// the caller's backward workspace and is zeroed by the preprocess kernel of the same call.
//
// Inside a CTA the roles (TMA producer, MMA issuer, elementwise warps) walk the same sequence
// of items, each at its own pace.  One thread (the producer's) fetches the ids and hands them
// on through a ring of kQueueSlots shared-memory slots: slot r % kQueueSlots holds round r's
// id, -1 once the work has run out; a full barrier per slot (one arrive: the fetch) and an
// empty barrier per slot (one arrive per consumer warp) order the hand-over.  The fetcher runs
// one round ahead of its own loads, so a consumer that looks one item ahead never waits for
// copies that wait on it.
#pragma once

#include "fa_ptx.cuh"

namespace fa {

constexpr int kQueueSlots = 4;

struct WorkQueue {
    uint64_t full[kQueueSlots], empty[kQueueSlots];
    int id[kQueueSlots];
};

// One thread, at set-up (before the CTA's first barrier): `consumer_warps` warps read each slot.
__device__ __forceinline__ void queue_init(WorkQueue& q, uint32_t consumer_warps) {
    for (int s = 0; s < kQueueSlots; ++s) {
        mbar_init(&q.full[s], 1);
        mbar_init(&q.empty[s], consumer_warps);
    }
}

// The fetching thread: publishes round `round`'s id (the next one from *counter, or -1 when
// the ids reach `total` or an earlier round already published -1) once its slot is free.
// Returns the id, or -2 when the wait for the slot gave up.
__device__ __forceinline__ int queue_push(WorkQueue& q, int round, int* counter, int total,
                                          bool exhausted, const volatile int* abort,
                                          uint64_t timeout_ns) {
    const int s = round % kQueueSlots;
    if (round >= kQueueSlots &&
        !wait_bounded(&q.empty[s], ((uint32_t)(round / kQueueSlots) - 1u) & 1u, abort,
                      timeout_ns))
        return -2;
    int id = -1;
    if (!exhausted) {
        id = atomicAdd(counter, 1);
        if (id >= total) id = -1;
    }
    *reinterpret_cast<volatile int*>(&q.id[s]) = id;
    mbar_arrive(&q.full[s]);  // release: the id is visible to the waiters
    return id;
}

// A consumer warp (all lanes): round `round`'s id (warp-uniform), or -2 when the wait gave
// up.  Lane 0 then frees the slot for the fetcher.
__device__ __forceinline__ int queue_pop_warp(WorkQueue& q, int round, const volatile int* abort,
                                              uint64_t timeout_ns) {
    const int s = round % kQueueSlots;
    if (!wait_warp(&q.full[s], (uint32_t)(round / kQueueSlots) & 1u, abort, timeout_ns))
        return -2;
    const int id = *reinterpret_cast<volatile int*>(&q.id[s]);
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&q.empty[s]);
    return id;
}

}  // namespace fa
