// Batched (chunked) prefill for dense bf16 models with head_dim 128.
#pragma once

#include <cuda.h>

#include <string>

#include "df_internal.h"

namespace df {

struct TcPlan;
struct AttnPlan;
struct MoePlan;

struct BpPlan {
  bool enabled = false;
  int mcap = 0;                 // activation rows per chunk (B x positions), a multiple of 128
  float* h = nullptr;           // [mcap][d] residual rows of the chunk
  void* u = nullptr;            // [mcap][d] normed rows (bf16)
  void* q = nullptr;            // [mcap][qdim] rotated queries (bf16)
  void* o = nullptr;            // [mcap][qdim] attention output (bf16)
  void* z = nullptr;            // [mcap][F] SwiGLU output (bf16)
  CUtensorMap x_u, x_o, x_z;    // activation maps, 128-row boxes
  // MoE layers: routing of the chunk's rows and the experts' packed blocks
  bool moe = false;
  int maxblk = 0;               // 128-row blocks the packed buffers hold
  float* un = nullptr;          // [mcap][d] normed rows, unrounded (router input)
  float* rlog = nullptr;        // [mcap][E] router logits
  int *sel_e = nullptr, *sel_slot = nullptr;  // [mcap][k] expert and slot of entry (m, j)
  float* sel_g = nullptr;       // [mcap][k] gates
  int *ecount = nullptr, *poff = nullptr, *gblk = nullptr;  // [E], [E], [maxblk][2]
  void* xg = nullptr;           // [maxblk * 128][d] packed expert inputs (bf16)
  void* zg = nullptr;           // [maxblk * 128][Fe] packed SwiGLU outputs (bf16)
  float* yg = nullptr;          // [maxblk * 128][d] packed expert outputs (fp32)
  CUtensorMap x_xg, x_zg;
};

// Rows per chunk for a model, or 0 when batched prefill does not apply
// (bf16, head_dim 128, 128-multiple widths; MoE: expert hidden a multiple of
// 64, at most 1024 experts and top_k <= 16).
int bp_rows(const Dims& D);
// Workspace bytes of the chunk buffers (0 when it does not apply).
size_t bp_workspace_bytes(const Dims& D);
// Carves the chunk buffers from `region` and encodes their tensor maps.
bool bp_init(BpPlan& P, const Dims& D, void* region, std::string* err);
// Prefill positions [0, n) of B sequences (primary flow only): tokens is a
// device [B][n] array of ids; sequence i of the call is cache sequence
// slot0 + i.  Every layer runs once per chunk of positions; the KV cache
// receives positions 0..n-1 (paged mode: into the pages the table already
// lists for them).  Enqueued on `s`.
// MoE models route through `moe` (its stacked expert weight maps) with the
// router matrices `router` ([L]).
void bp_prefill(const BpPlan& P, const TcPlan& tc, const AttnPlan& at, const MoePlan* moe, const Dims& D,
                const Buffers& Bf, void* kv, const void* emb1, const float* const* attn_norm,
                const float* const* mlp_norm, const void* const* router, const int32_t* tokens, int B, int n,
                int slot0, cudaStream_t s);

}  // namespace df
