// cluster_exit.cuh — the cluster barrier that the projection and decode kernels pass before
// leaving (device code).
#pragma once

namespace ea {

// A barrier over every thread of every CTA of the cluster, used only so that no CTA leaves (and
// gives back its shared memory) while a peer may still read it: the peers' loads have returned
// their values before they arrive, so the arrival needs no release, and a relaxed one does not
// wait for the arriving thread's own global stores.
__device__ __forceinline__ void cluster_sync_exit() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}

}  // namespace ea
