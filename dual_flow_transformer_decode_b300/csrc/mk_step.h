// Persistent decode-pass kernel for dense bf16 models: one launch runs every
// layer of a decode (or prefill) pass.  See mk_step.cu.
#pragma once

#include <cuda.h>

#include <string>
#include <vector>

#include "df_internal.h"

namespace df {

// One unit of work of one CTA, in the CTA's execution order.
struct MkTask {
  uint8_t type;    // MK_GEMM, MK_ATTN, MK_NORM
  uint8_t phase;   // GEMM: MK_QKV..MK_DN; NORM: 0 (before attention) or 1 (before the MLP)
  uint16_t layer;
  uint16_t tile;   // GEMM: 128-row weight tile; ATTN: (sequence, KV head) pair; NORM: stacked row
  uint16_t a0, a1; // GEMM: k-block range [a0, a1)
  uint8_t seg;     // GEMM/ATTN: segment index within the tile / pair
  uint8_t nseg;    // number of segments of that tile / pair
  uint32_t part;   // GEMM/ATTN: partial-result slot of this segment
};
static_assert(sizeof(MkTask) == 16, "MkTask layout");

enum : uint8_t { MK_GEMM = 0, MK_ATTN = 1, MK_NORM = 2 };
enum : uint8_t { MK_QKV = 0, MK_WO = 1, MK_GU = 2, MK_DN = 3 };

// Per-layer vectors the kernel reads directly.
struct MkLayer {
  const float *g1, *g2;     // RMSNorm gains before attention / before the MLP
  const float *a, *b, *c;   // couplings
};

// Task lists of one set of active stacked rows ([0,2B), [0,B) or [B,2B)).
struct MkRowSet {
  bool built = false;
  int lo = 0, hi = 0, N = 0;   // rows and the MMA N they are padded to
  int maxT = 0;                // task slots per CTA in the device list
  MkTask* tasks = nullptr;     // [sms][maxT]
  int* ntasks = nullptr;       // [sms]
  CUtensorMap* xmap = nullptr; // [3]: u (QKV, gate/up input), o (Wo input), z (down input)
};

struct MkPlan {
  bool enabled = false;
  int B = 0;
  int sms = 0;
  int max_tiles = 0;           // counter stride per (layer, phase)
  int maxT_cap = 0;
  CUtensorMap* wmap = nullptr; // [L][4]
  CUtensorMap* kvmap = nullptr;
  MkLayer* layers = nullptr;   // [L]
  uint8_t* tnseg = nullptr;    // [4][max_tiles]: segments per tile of each GEMM phase
  int segs[4] = {0, 0, 0, 0};  // segments per GEMM phase
  uint32_t* cnt = nullptr;     // dependency counters and tickets
  size_t ncnt = 0;
  float* gpart = nullptr;      // GEMM segment partials, one region per phase
  size_t gregion = 0;          // floats per phase region
  float* apart = nullptr;      // attention segment partials
  MkRowSet rs[3];              // 0: both flows, 1: primary rows, 2: auxiliary rows
  size_t smem = 0;
};

// Whether the persistent kernel is enabled (DF_MK=1) and supports the model
// (bf16, dense, head_dim 128, G <= 4, 128-multiple widths); `why` receives
// the reason when it is not.
bool mk_supported(const Dims& D, std::string* why);
// Workspace bytes the plan needs: reserved for every model of supported
// shape, enabled or not, so the size does not depend on the environment.
size_t mk_workspace_bytes(const Dims& D);
// Carves the plan's buffers from `region` and encodes the weight and cache
// tensor maps.  Leaves P.enabled false when unsupported or disabled.
bool mk_init(MkPlan& P, const Dims& D, const Buffers& Bf, void* region, void* kv,
             const std::vector<const void*>& wqkv, const std::vector<const void*>& wo,
             const std::vector<const void*>& wgu, const std::vector<const void*>& wd,
             const std::vector<const float*>& g1, const std::vector<const float*>& g2,
             const std::vector<const float*>& a, const std::vector<const float*>& b,
             const std::vector<const float*>& c, cudaStream_t s, std::string* err);
// Builds the task lists for batch B (synchronous host-to-device copies).
bool mk_batch(MkPlan& P, const Dims& D, const Buffers& Bf, int B, std::string* err);
bool mk_can_run(const MkPlan& P, const Rows& R);
// Floats of attention segment partials a launch may write (the capacity of
// the plan's region: every row set, every segment count the planner picks).
size_t mk_attn_partial_floats(const Dims& D);
// One launch: every layer of a pass over rows R.
void mk_launch(const MkPlan& P, const Dims& D, const Buffers& Bf, void* kv, const Rows& R, int save, int saved,
               cudaStream_t s);

}  // namespace df
