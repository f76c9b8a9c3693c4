// Ranks of routed (token, slot) pairs inside a block of tokens, for the
// dispatch's stable permutation (expert ascending, then token ascending):
// the mma router computes them while the ids are still at hand, so the
// dispatch only has to add per-block bases.
#pragma once
#include <cstdint>

namespace cbmoe {

// Lane l holds token l of a group of up to 32 consecutive tokens (valid =
// false for lanes past the end) with k distinct expert ids ids[0..k).  For
// each slot s, rank[s] = counts[e] + #{lanes l' < l whose ids contain e},
// e = ids[s]; then counts[e] (shared memory, updated by lane 0) grows by
// #{lanes whose ids contain e}.  Called for consecutive groups in token
// order, counts[e] runs over the whole block.  One ballot per expert: E
// iterations of k compares.
template <int KMAX>
__device__ __forceinline__ void warp_expert_ranks(const int (&ids)[KMAX], int k, bool valid, int E, int* counts,
                                                  int (&rank)[KMAX]) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int s = 0; s < KMAX; ++s) rank[s] = 0;
  for (int e = 0; e < E; ++e) {
    bool mine = false;
#pragma unroll
    for (int s = 0; s < KMAX; ++s) mine = mine || (s < k && ids[s] == e);
    mine = mine && valid;
    const uint32_t b = __ballot_sync(0xffffffffu, mine);
    if (b == 0u) continue;  // uniform across the warp
    const int prior = counts[e];
    __syncwarp();
    if (mine) {
      const int r = prior + __popc(b & lt);
#pragma unroll
      for (int s = 0; s < KMAX; ++s)
        if (s < k && ids[s] == e) rank[s] = r;
    }
    if (lane == 0) counts[e] = prior + __popc(b);
    __syncwarp();
  }
}

}  // namespace cbmoe
