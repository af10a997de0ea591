// topk_plan.h -- which top-K plans finish their rows inside the chunk kernel.
// Rows of 2, 4 or 8 chunks run as one thread-block cluster per row whose
// first CTA merges the others' candidates from their shared memory: no merge
// kernel and no workspace. A row of one chunk is finished by its own CTA.
// Other chunk counts go through the merge kernel.
#pragma once

namespace fa {

constexpr int kTopkMaxCluster = 8;

inline bool topk_clustered(int n_chunks) {
  return n_chunks == 1 || n_chunks == 2 || n_chunks == 4 || n_chunks == kTopkMaxCluster;
}

}  // namespace fa
