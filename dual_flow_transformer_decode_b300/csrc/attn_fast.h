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
};

bool attn_fast_init(AttnPlan& P, const Dims& D, void* kv, std::string* err);
void attn_fast_free(AttnPlan& P);
bool attn_fast_can_run(const AttnPlan& P, const Dims& D);
void attn_fast(const AttnPlan& P, const Dims& D, const Buffers& Bf, const void* kv, int layer, int splits,
               const Rows& R, cudaStream_t s);

}  // namespace df
