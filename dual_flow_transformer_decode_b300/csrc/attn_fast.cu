// Fast shared-KV attention: placeholder until the TMA kernel lands.
#include "attn_fast.h"

namespace df {

bool attn_fast_init(AttnPlan& P, const Dims&, void*, std::string*) {
  P.enabled = false;
  return true;
}
void attn_fast_free(AttnPlan&) {}
bool attn_fast_can_run(const AttnPlan& P, const Dims&) { return P.enabled; }
void attn_fast(const AttnPlan&, const Dims&, const Buffers&, const void*, int, int, const Rows&, cudaStream_t) {}

}  // namespace df
