// Tensor-core (tcgen05 + TMEM, TMA-fed) GEMMs with fused epilogues.
#pragma once

#include <cuda.h>
#include <string>
#include <vector>

#include "df_internal.h"

namespace df {

enum class TcOp { QKV = 0, RESID = 1, SWIGLU = 2, DOWN = 3, LOGITS = 4 };

struct TcPlan {
  bool enabled = false;
  int B = 0;
  int npad = 0;                // stacked rows padded to the MMA N granule
  int sms = 0;                 // streaming multiprocessors of the device
  int splits[5] = {1, 1, 1, 1, 1};
  bool dense = true;
  int mpad = 0;                // rows allocated in the activation buffers
  void *u_ptr = nullptr, *o_ptr = nullptr, *z_ptr = nullptr;
  std::vector<CUtensorMap> w_qkv, w_o, w_gu, w_d;
  CUtensorMap w_lm;
  CUtensorMap x_u, x_o, x_z;
  // Failure-detection test hook: DF_TEST_GEMM_STALL_NS at df_create makes
  // every GEMM launch let one bounded wait run out (see k_tc_gemm).
  unsigned long long stall_ns = 0;
  // Stacked rows up to which the small projections run as a CUDA-core GEMV
  // instead of tensor-core tiles (measured crossover: 2; DF_GEMV_ROWS
  // overrides, at most 8), and which ops of this batch take it.
  int gemv_max_rows = 2;
  bool gemv[5] = {false, false, false, false, false};
};

size_t tc_tickets_needed(const Dims& D);
size_t tc_partial_floats(const Dims& D);
bool tc_plan_init(TcPlan& P, const Dims& D, const Buffers& Bf, const std::vector<const void*>& wqkv,
                  const std::vector<const void*>& wo, const std::vector<const void*>& wgu,
                  const std::vector<const void*>& wd, const void* lm_head, std::string* err);
bool tc_plan_batch(TcPlan& P, const Dims& D, int B, std::string* err);
void tc_plan_free(TcPlan& P);
bool tc_can_run(const TcPlan& P, TcOp op);

void tc_qkv(const TcPlan& P, const Dims& D, const Buffers& Bf, const void* w, const float* a, void* kv, int layer,
            const Couple& C, const Rows& R, cudaStream_t s);
void tc_resid(const TcPlan& P, const Dims& D, const Buffers& Bf, const void* w, int layer, const Rows& R,
              cudaStream_t s);
void tc_swiglu(const TcPlan& P, const Dims& D, const Buffers& Bf, const void* w, int layer, const float* bvec,
               const Couple& C, const Rows& R, cudaStream_t s);
void tc_down(const TcPlan& P, const Dims& D, const Buffers& Bf, const void* w, int layer, const float* cvec,
             const Couple& C, const Rows& R, cudaStream_t s);
void tc_logits(const TcPlan& P, const Dims& D, const Buffers& Bf, const void* w, const Rows& R, cudaStream_t s);

}  // namespace df
