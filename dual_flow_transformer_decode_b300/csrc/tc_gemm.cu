// Tensor-core GEMMs: placeholder until the tcgen05 kernels land.
#include "tc_gemm.h"

namespace df {

size_t tc_tickets_needed(const Dims&) { return 1; }
size_t tc_partial_floats(const Dims&) { return 1; }
bool tc_plan_init(TcPlan& P, const Dims&, const Buffers&, const std::vector<const void*>&,
                  const std::vector<const void*>&, const std::vector<const void*>&,
                  const std::vector<const void*>&, const void*, std::string*) {
  P.enabled = false;
  return true;
}
bool tc_plan_batch(TcPlan& P, const Dims&, int B, std::string*) {
  P.B = B;
  return true;
}
void tc_plan_free(TcPlan&) {}
bool tc_can_run(const TcPlan& P, TcOp) { return P.enabled; }
void tc_qkv(const TcPlan&, const Dims&, const Buffers&, const void*, const float*, void*, int, const Couple&,
            const Rows&, cudaStream_t) {}
void tc_resid(const TcPlan&, const Dims&, const Buffers&, const void*, const Rows&, cudaStream_t) {}
void tc_swiglu(const TcPlan&, const Dims&, const Buffers&, const void*, const float*, const Couple&, const Rows&,
               cudaStream_t) {}
void tc_down(const TcPlan&, const Dims&, const Buffers&, const void*, const float*, const Couple&, const Rows&,
             cudaStream_t) {}
void tc_logits(const TcPlan&, const Dims&, const Buffers&, const void*, const Rows&, cudaStream_t) {}

}  // namespace df
