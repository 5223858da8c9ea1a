// Split-KV shared-KV decode attention for head_dim 128 bf16 caches:
// TMA-staged K/V tiles serve the primary and auxiliary queries of a KV head.
#pragma once

#include <cuda.h>
#include <string>

#include "df_internal.h"

namespace df {

struct AttnPlan {
  bool enabled = false;
  CUtensorMap kv;   // 3-D view: (head_dim, positions of a page, L*2*pages*Hkv)
  // clusters of s CTAs (one per KV split) that the device holds at once,
  // from the occupancy query at init; 0 when unknown
  int max_clusters[17] = {};
};

bool attn_fast_init(AttnPlan& P, const Dims& D, void* kv, std::string* err);
void attn_fast_free(AttnPlan& P);
bool attn_fast_can_run(const AttnPlan& P, const Dims& D);
// KV splits per (sequence, KV head) for batch B: the time model of
// attn_splits with the waves counted from the measured cluster capacity.
int attn_fast_splits(const AttnPlan& P, const Dims& D, int B);
void attn_fast(const AttnPlan& P, const Dims& D, const Buffers& Bf, const void* kv, int layer, int splits,
               const Rows& R, cudaStream_t s);

}  // namespace df
