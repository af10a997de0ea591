// topk_plan.h -- which top-K plans finish their rows inside the chunk kernel.
// A row of one chunk is finished by its own CTA. For K up to
// kTopkClusterMaxK (two chunk CTAs share an SM), rows of 2, 4 or 8 chunks run
// as one thread-block cluster per row whose first CTA merges the others'
// candidates from their shared memory: no merge kernel and no workspace.
// Larger K (one CTA per SM: a cluster would have to find that many free SMs
// in one GPC, stranding the rest) and other chunk counts go through the
// merge kernel.
#pragma once

namespace fa {

constexpr int kTopkMaxCluster = 8;
constexpr int kTopkClusterMaxK = 128;

inline bool topk_clustered(int n_chunks, int K) {
  if (n_chunks == 1) return true;
  return K <= kTopkClusterMaxK &&
         (n_chunks == 2 || n_chunks == 4 || n_chunks == kTopkMaxCluster);
}

}  // namespace fa
