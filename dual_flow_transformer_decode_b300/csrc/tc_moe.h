// Tensor-core grouped expert GEMMs of the MoE layer (router replay).
#pragma once

#include <cuda.h>
#include <string>
#include <vector>

#include "df_internal.h"

namespace df {

struct MoePlan {
  bool enabled = false;
  int nxe = 0;     // rows of one expert's packed block: 2 * max_batch padded to 16
  int stages = 0;  // TMA ring depth of the expert GEMMs
  std::vector<CUtensorMap> w_gu, w_d;
  CUtensorMap x_g, x_z;
};

int moe_nxe(const Dims& D);
bool moe_tc_init(MoePlan& P, const Dims& D, const Buffers& Bf, const std::vector<const void*>& wgu,
                 const std::vector<const void*>& wd, std::string* err);
void moe_tc_free(MoePlan& P);
// Gather, gate/up + SwiGLU + b, down, combine + c + residual (routing done).
// With next_norm set, the combine also writes the RMSNorm of the updated
// rows with those gains into u (the next layer's attention norm, or the
// final norm), in the same launch.
void moe_tc_forward(const MoePlan& P, const Dims& D, const Buffers& Bf, int layer, const float* bvec,
                    const float* cvec, const Couple& C, const Rows& R, cudaStream_t s,
                    const float* next_norm = nullptr);

}  // namespace df
