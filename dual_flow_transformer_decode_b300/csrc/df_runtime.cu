// C-ABI runtime of the dual-flow decode library: configuration checks,
// workspace layout, the per-step kernel sequence, CUDA-graph capture and
// replay, and device error reporting.
//
// Step sequence ("Arquitectura Central" and "Mecanismos Clave" of "Resumen
// Técnico: Dual-Flow Transformers"):
//   prefill position:  embed(primary) -> per layer [norm, QKV+RoPE+append,
//                      attention, Wo+residual, norm, MLP] -> advance t
//   grouped decode:    embed(both flows, stacked) -> per layer the same chain
//                      over 2B rows with the a/b/c couplings in the epilogues
//                      -> final norm -> LM head -> mixture -> advance t
//   ungrouped decode:  the same layers run once for the primary rows (saving
//                      q1, z1, y1) and once more for the auxiliary rows.

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "df.h"
#include "df_internal.h"
#include "tc_gemm.h"
#include "tc_moe.h"
#include "attn_fast.h"
#include "mk_step.h"
#include "prefill.h"

using df::Buffers;
using df::Couple;
using df::Dims;
using df::Rows;

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct GraphKey {
  const void* p[8];
  int i[6];
  bool operator==(const GraphKey& o) const {
    return memcmp(p, o.p, sizeof(p)) == 0 && memcmp(i, o.i, sizeof(i)) == 0;
  }
};

struct GraphSlot {
  bool valid = false;
  GraphKey key{};
  cudaGraphExec_t exec = nullptr;
  int kernels = 0;
  void reset() {
    if (exec) cudaGraphExecDestroy(exec);
    exec = nullptr;
    valid = false;
  }
};

}  // namespace

struct df_ctx {
  df_config cfg{};
  Dims D{};
  Buffers Bf{};
  const void *emb1 = nullptr, *emb2 = nullptr, *lm_head = nullptr;
  const float* final_norm = nullptr;
  std::vector<const float*> attn_norm, mlp_norm, a, b, c;
  std::vector<const void*> wqkv, wo, wgu, wd, router;
  void* kv = nullptr;
  char* ws = nullptr;
  cudaStream_t stream = nullptr;
  bool own_stream = false;
  int B = 0, t = 0, splits = 1;
  int splits_fast = 1;  // KV splits of the TMA attention kernel (cluster-capacity aware)
  bool ready = false;
  int aux_on = 1, ungrouped = 0;
  float *dbg_logp1 = nullptr, *dbg_logp2 = nullptr, *dbg_router = nullptr;
  int32_t* dbg_topk = nullptr;
  bool use_graph = true;
  int force_generic = 0;
  GraphSlot dec, pre;
  GraphSlot dec_static;  // graph of df_decode_step_noalloc
  GraphSlot gen;         // graph of one df_generate step
  // pipelined host-buffer steps: output copies on their own stream, from two
  // staging areas used in turn (each with its own captured step graph)
  GraphSlot dec_host[2];
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t step_done[2] = {nullptr, nullptr}, copy_done[2] = {nullptr, nullptr};
  int host_slot = 0;
  int last_kernels = -1;
  df::TcPlan tc;
  df::MoePlan moe;
  df::AttnPlan at;
  df::MkPlan mk;
  df::BpPlan bp;
  std::string err;
  // paged mode: the page pool as the host tracks it (the device table and
  // positions mirror it; every change is enqueued before the work that
  // depends on it)
  std::vector<int> free_pages;              // stack of free physical pages
  std::vector<std::vector<int>> seq_pages;  // per slot: physical page of each logical page
  std::vector<int> seq_len;                 // per slot: length, -1 for a free slot
};

namespace {

df_status fail(df_ctx* X, df_status st, const std::string& msg) {
  if (X) X->err = msg;
  return st;
}

df_status cuda_fail(df_ctx* X, cudaError_t e, const char* where) {
  return fail(X, DF_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

bool valid_config(const df_config* c, std::string* why) {
  auto bad = [&](const char* m) {
    if (why) *why = m;
    return false;
  };
  if (!c) return bad("null config");
  if (c->n_layers <= 0 || c->d_model <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 ||
      c->vocab <= 0)
    return bad("non-positive model size");
  if (c->n_heads % c->n_kv_heads) return bad("n_heads must be a multiple of n_kv_heads");
  if (c->head_dim % 2) return bad("head_dim must be even (RoPE pairs)");
  if (c->d_model % 8 || c->d_model > 8192) return bad("d_model must be a multiple of 8 and at most 8192");
  if (c->dtype != DF_F32 && c->dtype != DF_BF16) return bad("dtype must be DF_F32 or DF_BF16");
  if (c->max_batch <= 0 || c->max_len <= 0) return bad("max_batch and max_len must be positive");
  if (c->max_batch > 4096) return bad("max_batch above 4096");
  if (c->n_experts < 0) return bad("n_experts < 0");
  if (c->n_experts == 0) {
    if (c->ffn_hidden <= 0 || c->ffn_hidden % 64) return bad("ffn_hidden must be a positive multiple of 64");
  } else {
    if (c->top_k <= 0 || c->top_k > c->n_experts || c->top_k > 16) return bad("top_k must be in [1, min(16, E)]");
    if (c->expert_hidden <= 0 || c->expert_hidden % 64) return bad("expert_hidden must be a positive multiple of 64");
    if (c->aux_top_k && (c->aux_top_k < c->top_k || c->aux_top_k > c->n_experts || c->aux_top_k > 16))
      return bad("aux_top_k must be 0 or in [top_k, min(16, E)]");
  }
  if (c->n_experts > 4096) return bad("n_experts above 4096");
  if (!(c->norm_eps > 0.f) || !(c->rope_theta > 0.f)) return bad("norm_eps and rope_theta must be positive");
  if (c->page_len) {
    if (c->page_len < 64 || c->page_len > (1 << 20) || (c->page_len & (c->page_len - 1)))
      return bad("page_len must be 0 or a power of two in [64, 2^20]");
    if (c->n_pages <= 0) return bad("n_pages must be positive in paged mode");
    // tensor-map rows of the cache: n_layers * 2 * (n_pages + 1) * n_kv_heads
    if ((double)c->n_layers * 2 * ((double)c->n_pages + 1) * c->n_kv_heads >= 2147483647.0)
      return bad("page pool too large");
  } else if (c->n_pages) {
    return bad("n_pages needs page_len");
  }
  return true;
}

Dims make_dims(const df_config* c) {
  Dims D{};
  D.L = c->n_layers;
  D.d = c->d_model;
  D.Hq = c->n_heads;
  D.Hkv = c->n_kv_heads;
  D.hd = c->head_dim;
  D.F = c->n_experts ? 0 : c->ffn_hidden;
  D.V = c->vocab;
  D.E = c->n_experts;
  D.k = c->n_experts ? c->top_k : 0;
  D.ka = c->n_experts ? (c->aux_top_k > c->top_k ? c->aux_top_k : c->top_k) : 0;
  D.Fe = c->n_experts ? c->expert_hidden : 0;
  D.theta = c->rope_theta;
  D.eps = c->norm_eps;
  D.bf16 = c->dtype == DF_BF16;
  D.maxB = c->max_batch;
  D.max_len = c->max_len;
  D.qdim = D.Hq * D.hd;
  D.kvdim = D.Hkv * D.hd;
  D.qkvn = D.qdim + 2 * D.kvdim;
  D.G = D.Hq / D.Hkv;
  D.Fm = D.E ? D.Fe : D.F;
  D.esz = D.bf16 ? 2 : 4;
  if (c->page_len) {
    D.paged = 1;
    D.PG = c->page_len;
    D.NP = c->n_pages + 1;  // the last page is the sink of free slots
    // one more column than the positions need: a full sequence (position
    // max_len) still maps to an entry, the sink
    D.MPS = D.max_len / D.PG + 1;
    D.pg_shift = 0;
    while ((1 << D.pg_shift) < D.PG) ++D.pg_shift;
  } else {
    D.paged = 0;
    D.PG = D.max_len;
    D.NP = D.maxB;
    D.MPS = 1;
    D.pg_shift = 0;
  }
  // the split plan and workspace size depend on the SM count of the current device
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 148;
  D.sms = sms;
  return D;
}

// Carves the workspace.  With base == nullptr only the size is computed.
size_t layout(const Dims& D, Buffers* Bf, char* base) {
  size_t cur = 0;
  auto take = [&](size_t bytes) -> char* {
    size_t o = cur;
    cur = align_up(cur + (bytes ? bytes : 1), 256);
    return base ? base + o : nullptr;
  };
  size_t M2 = 2 * (size_t)D.maxB, Mpad = align_up(M2, 16);
  size_t esz = D.esz;
  Buffers b{};
  b.ctrl = (df::Ctrl*)take(sizeof(df::Ctrl));
  b.kv_table = (int*)take(D.paged ? (size_t)D.maxB * D.MPS * 4 : 0);
  b.kv_pos = (int*)take((size_t)D.maxB * 4);
  b.kv_active = (int*)take((size_t)D.maxB * 4);
  b.kvm = df::KvMap{D.paged ? b.kv_table : nullptr, b.kv_pos, b.kv_active, D.NP, D.PG, D.MPS, D.pg_shift};
  b.tokbuf = (int*)take(D.maxB * 4);
  b.h = (float*)take(M2 * D.d * 4);
  b.u = take(Mpad * D.d * esz);
  b.un = (float*)take(D.E ? M2 * D.d * 4 : 0);
  b.qatt = (float*)take(M2 * D.qdim * 4);
  b.o = take(Mpad * D.qdim * esz);
  b.z = take(Mpad * (size_t)D.F * esz);
  size_t rawN = D.qkvn;
  if ((size_t)2 * D.F > rawN) rawN = 2 * D.F;
  if ((size_t)D.d > rawN) rawN = D.d;
  if ((size_t)D.E > rawN) rawN = D.E;
  b.rawN = (int)rawN;
  b.raw = (float*)take(Mpad * rawN * 4);
  b.logits = (float*)take(M2 * D.V * 4);
  b.gpart = (float*)take(df::tc_partial_floats(D) * 4);
  size_t parts = 0;
  for (int B = 1; B <= D.maxB; ++B) {
    size_t p = (size_t)B * D.Hkv * df::attn_splits(D, B) * 2 * D.G;
    if (p > parts) parts = p;
  }
  b.parts_cap = parts;
  b.part_o = (float*)take(parts * D.hd * 4);
  b.part_ml = (float*)take(parts * 2 * 4);
  size_t zs = D.E ? (size_t)D.k * D.Fe : (size_t)D.F;
  b.q1s = (float*)take((size_t)D.L * D.maxB * D.qdim * 4);
  b.z1s = (float*)take((size_t)D.L * D.maxB * zs * 4);
  b.y1s = (float*)take((size_t)D.L * D.maxB * D.d * 4);
  b.topk = (int*)take(D.E ? (size_t)D.L * D.maxB * D.k * 4 : 0);
  b.gate = (float*)take(D.E ? M2 * D.ka * 4 : 0);
  b.topkx = (int*)take(D.E ? (size_t)D.maxB * (D.ka - D.k) * 4 : 0);
  b.ecount = (int*)take(D.E * 4);
  b.elist = (int*)take((size_t)D.E * D.maxB * 4);
  b.zE = take(D.E ? 2 * (size_t)D.maxB * D.ka * D.Fe * esz : 0);
  b.yE = (float*)take(D.E ? 2 * (size_t)D.maxB * D.ka * D.d * 4 : 0);
  b.eslot = (int*)take(D.E ? (size_t)D.maxB * D.ka * 4 : 0);
  b.ticket = (int*)take(D.E ? 16 : 0);
  const size_t nxe = D.E ? (size_t)df::moe_nxe(D) : 0;
  b.xg = take(D.E * nxe * D.d * esz);
  b.zEt = take(D.E * nxe * D.Fe * esz);
  b.yEt = (float*)take(D.E * nxe * D.d * 4);
  b.out_logp = (float*)take((size_t)D.maxB * D.V * 4);
  b.out_arg = (int*)take(D.maxB * 4);
  b.out_alpha = (float*)take(D.maxB * 4);
  b.out_logp2 = (float*)take((size_t)D.maxB * D.V * 4);
  b.out_arg2 = (int*)take(D.maxB * 4);
  b.out_alpha2 = (float*)take(D.maxB * 4);
  b.gen_tok = (int*)take(D.maxB * 4);
  b.gen_hist = (int*)take((size_t)D.max_len * D.maxB * 4);
  b.rope = (float*)take((size_t)(D.max_len + 1) * D.hd * 4);
  b.mk_bytes = df::mk_workspace_bytes(D);
  b.mk = b.mk_bytes ? take(b.mk_bytes) : nullptr;
  b.bp_bytes = df::bp_workspace_bytes(D);
  b.bp = b.bp_bytes ? take(b.bp_bytes) : nullptr;
  if (Bf) *Bf = b;
  return cur;
}

size_t kv_size(const Dims& D) { return (size_t)D.L * D.kv_layer_elems() * D.esz; }

// ---------------------------------------------------------------- step sequencing

struct StepOut {
  float* logp_mix;
  int32_t* argmax;
  float* alpha;
  int32_t* sample_tok = nullptr;   // generation: the drawn tokens, the next step's input
  int32_t* sample_hist = nullptr;  // generation: [max_len][maxB] history of draws
};

Couple layer_couple(df_ctx* X, int l, int save, int saved) {
  const Dims& D = X->D;
  const Buffers& Bf = X->Bf;
  size_t zs = D.E ? (size_t)D.k * D.Fe : (size_t)D.F;
  return Couple{saved, save, Bf.q1s + (size_t)l * D.maxB * D.qdim, Bf.z1s + (size_t)l * D.maxB * zs,
                Bf.y1s + (size_t)l * D.maxB * D.d};
}

// QKV projection + Q2 coupling + RoPE + cache append (input: normed rows u).
void op_qkv(df_ctx* X, int l, const Rows& R, const Couple& C) {
  const Dims& D = X->D;
  const Buffers& Bf = X->Bf;
  if (!X->force_generic && df::tc_can_run(X->tc, df::TcOp::QKV)) {
    df::tc_qkv(X->tc, D, Bf, X->wqkv[l], X->a[l], X->kv, l, C, R, X->stream);
  } else {
    df::launch_gemv(D, X->wqkv[l], D.qkvn, D.d, Bf.u, D.d, Bf.raw, Bf.rawN, R, X->stream);
    df::launch_ep_qkv(D, Bf, Bf.raw, Bf.rawN, X->a[l], X->kv, l, C, R, X->stream);
  }
}

// Shared-KV attention of the active query rows, then the split merge.
void op_attn(df_ctx* X, int l, const Rows& R) {
  const Dims& D = X->D;
  if (!X->force_generic && df::attn_fast_can_run(X->at, D)) {
    df::attn_fast(X->at, D, X->Bf, X->kv, l, X->splits_fast, R, X->stream);  // merges its splits itself
  } else {
    df::launch_attention_generic(D, X->Bf, X->kv, l, X->splits, R, X->stream);
    df::launch_attn_combine(D, X->Bf, X->splits, R, X->stream);
  }
}

// Output projection + residual.
void op_wo(df_ctx* X, int l, const Rows& R) {
  const Dims& D = X->D;
  const Buffers& Bf = X->Bf;
  if (!X->force_generic && df::tc_can_run(X->tc, df::TcOp::RESID)) {
    df::tc_resid(X->tc, D, Bf, X->wo[l], l, R, X->stream);
  } else {
    df::launch_gemv(D, X->wo[l], D.d, D.qdim, Bf.o, D.qdim, Bf.raw, Bf.rawN, R, X->stream);
    df::launch_ep_residual(D, Bf, Bf.raw, Bf.rawN, R, X->stream);
  }
}

// Dense MLP, first half: gate/up + SwiGLU + b coupling.
void op_gateup(df_ctx* X, int l, const Rows& R, const Couple& C) {
  const Dims& D = X->D;
  const Buffers& Bf = X->Bf;
  if (!X->force_generic && df::tc_can_run(X->tc, df::TcOp::SWIGLU)) {
    df::tc_swiglu(X->tc, D, Bf, X->wgu[l], l, X->b[l], C, R, X->stream);
  } else {
    df::launch_gemv(D, X->wgu[l], 2 * D.F, D.d, Bf.u, D.d, Bf.raw, Bf.rawN, R, X->stream);
    df::launch_ep_swiglu(D, Bf, Bf.raw, Bf.rawN, X->b[l], C, R, X->stream);
  }
}

// Dense MLP, second half: down + c coupling + residual.
void op_down(df_ctx* X, int l, const Rows& R, const Couple& C) {
  const Dims& D = X->D;
  const Buffers& Bf = X->Bf;
  if (!X->force_generic && df::tc_can_run(X->tc, df::TcOp::DOWN)) {
    df::tc_down(X->tc, D, Bf, X->wd[l], l, X->c[l], C, R, X->stream);
  } else {
    df::launch_gemv(D, X->wd[l], D.d, D.F, Bf.z, D.F, Bf.raw, Bf.rawN, R, X->stream);
    df::launch_ep_down(D, Bf, Bf.raw, Bf.rawN, X->c[l], C, R, X->stream);
  }
}

// MoE MLP with router replay (input: normed rows u and unrounded un).  With
// next_norm set and the tensor-core path taken, the combine also writes the
// RMSNorm of the updated rows with those gains into u; returns whether it
// did.
bool op_moe(df_ctx* X, int l, const Rows& R, const Couple& C, const float* next_norm = nullptr) {
  const Dims& D = X->D;
  const Buffers& Bf = X->Bf;
  cudaStream_t s = X->stream;
  df::launch_router_route(D, Bf, X->router[l], l, R.has_primary() ? 1 : 0, R, X->dbg_topk, X->dbg_router, s);
  if (!X->force_generic && X->moe.enabled) {
    df::moe_tc_forward(X->moe, D, Bf, l, X->b[l], X->c[l], C, R, s, next_norm);
    return next_norm != nullptr;
  } else {
    df::launch_moe_gateup_generic(D, Bf, X->wgu[l], X->b[l], C, R, s);
    df::launch_moe_down_generic(D, Bf, X->wd[l], R, s);
    df::launch_moe_combine(D, Bf, X->c[l], C, R, s);
  }
  return false;
}

// LM head over the final-normed rows.
void op_lm(df_ctx* X, const Rows& R) {
  const Dims& D = X->D;
  const Buffers& Bf = X->Bf;
  if (!X->force_generic && df::tc_can_run(X->tc, df::TcOp::LOGITS)) {
    df::tc_logits(X->tc, D, Bf, X->lm_head, R, X->stream);
  } else {
    df::launch_gemv(D, X->lm_head, D.V, D.d, Bf.u, D.d, Bf.logits, D.V, R, X->stream);
  }
}

// Every layer of a pass over rows R: one persistent-kernel launch where it
// applies, else the kernel sequence per layer.  lm_norm: the final norm's
// gains when the pass ends with the LM head (a fused MoE combine may then
// apply it); returns whether the final norm was applied.
bool enqueue_layers(df_ctx* X, const Rows& R, int save, int saved, const float* lm_norm = nullptr) {
  const Dims& D = X->D;
  const Buffers& Bf = X->Bf;
  cudaStream_t s = X->stream;
  if (!X->force_generic && df::mk_can_run(X->mk, R)) {
    df::mk_launch(X->mk, D, Bf, X->kv, R, save, saved, s);
    return false;
  }
  bool normed = false;  // u already holds this layer's attention-normed rows
  for (int l = 0; l < D.L; ++l) {
    Couple C = layer_couple(X, l, save, saved);
    if (!normed) df::launch_rmsnorm(D, Bf, X->attn_norm[l], Bf.u, nullptr, R, s);
    normed = false;
    op_qkv(X, l, R, C);
    op_attn(X, l, R);
    op_wo(X, l, R);
    df::launch_rmsnorm(D, Bf, X->mlp_norm[l], Bf.u, D.E ? Bf.un : nullptr, R, s);
    if (D.E) {
      normed = op_moe(X, l, R, C, l + 1 < D.L ? X->attn_norm[l + 1] : lm_norm);
    } else {
      op_gateup(X, l, R, C);
      op_down(X, l, R, C);
    }
  }
  return normed;
}

void enqueue_pass(df_ctx* X, const Rows& R, int save, int saved, bool lm) {
  const Dims& D = X->D;
  const Buffers& Bf = X->Bf;
  cudaStream_t s = X->stream;
  const bool normed = enqueue_layers(X, R, save, saved, lm ? X->final_norm : nullptr);
  if (lm) {
    if (!normed) df::launch_rmsnorm(D, Bf, X->final_norm, Bf.u, nullptr, R, s);
    op_lm(X, R);
  }
}

void enqueue_decode(df_ctx* X, const int32_t* tokens, const StepOut& o) {
  const Dims& D = X->D;
  int B = X->B;
  cudaStream_t s = X->stream;
  Rows both{B, 0, X->aux_on ? 2 * B : B};
  df::launch_embed(D, X->Bf, X->emb1, X->emb2, tokens, 1, 0, both, s);
  if (X->aux_on && X->ungrouped) {
    enqueue_pass(X, Rows{B, 0, B}, 1, 0, true);
    enqueue_pass(X, Rows{B, B, 2 * B}, 0, 1, true);
  } else {
    enqueue_pass(X, both, 0, 0, true);
  }
  df::launch_mix(D, X->Bf, B, X->aux_on, o.logp_mix, o.argmax, o.alpha, X->dbg_logp1, X->aux_on ? X->dbg_logp2 : nullptr,
                 o.sample_tok, o.sample_hist, s);
  df::launch_advance_pos(X->Bf, 0, B, s);
}

// One token-serial prefill position over all B primary rows.  Row b embeds
// tokens[b*stride + step] (step = the pass counter, reset before the first
// position); positions advance for the sequences [adv_lo, adv_hi) only.
void enqueue_prefill_pos(df_ctx* X, const int32_t* tokens, int stride, int adv_lo, int adv_hi) {
  Rows R{X->B, 0, X->B};
  df::launch_embed(X->D, X->Bf, X->emb1, X->emb2, tokens, stride, 1, R, X->stream);
  enqueue_pass(X, R, 0, 0, false);
  df::launch_advance_pos(X->Bf, adv_lo, adv_hi, X->stream);
}

// ------------------------------------------------------------------ paged mode

// Writes into one device int array (page table, positions or active flags),
// queued and flushed as small kernels on the context's stream.
struct EditQueue {
  df_ctx* X;
  int* dst;
  df::IntEdits e{};
  void add(int idx, int val) {
    if (e.n == df::kIntEdits) flush();
    e.idx[e.n] = idx;
    e.val[e.n] = val;
    ++e.n;
  }
  void flush() {
    df::launch_int_edits(dst, e, X->stream);
    e.n = 0;
  }
};

int pages_for(const Dims& D, int n) { return (n + D.PG - 1) / D.PG; }

// Returns slot b's pages to the pool and points its table row at the sink.
void release_slot(df_ctx* X, int b, EditQueue& tq) {
  auto& pg = X->seq_pages[b];
  for (int i = (int)pg.size() - 1; i >= 0; --i) {
    X->free_pages.push_back(pg[i]);
    tq.add(b * X->D.MPS + i, X->D.NP - 1);
  }
  pg.clear();
  X->seq_len[b] = -1;
}

// Maps positions [0, n) of slot b, taking pages from the pool; false (and
// nothing taken) when the pool is short.
bool grow_slot(df_ctx* X, int b, int n, EditQueue& tq) {
  auto& pg = X->seq_pages[b];
  const int need = pages_for(X->D, n) - (int)pg.size();
  if (need > (int)X->free_pages.size()) return false;
  for (int i = 0; i < need; ++i) {
    const int p = X->free_pages.back();
    X->free_pages.pop_back();
    tq.add(b * X->D.MPS + (int)pg.size(), p);
    pg.push_back(p);
  }
  return true;
}

// Before n decode steps: capacity checks (nothing enqueued on failure), then
// the pages the steps will write are mapped.  Contiguous mode: the common
// position must leave room for n steps.
df_status prepare_steps(df_ctx* X, int n, const char* who) {
  const Dims& D = X->D;
  if (!D.paged) {
    if (n > X->cfg.max_len - X->t) return fail(X, DF_ERR_CAPACITY, std::string(who) + ": cache full (t + steps > max_len)");
    return DF_OK;
  }
  int need = 0;
  for (int b = 0; b < X->B; ++b) {
    const int len = X->seq_len[b];
    if (len < 0) continue;
    if (n > X->cfg.max_len - len)
      return fail(X, DF_ERR_CAPACITY, std::string(who) + ": sequence " + std::to_string(b) + " would pass max_len");
    need += std::max(0, pages_for(D, len + n) - (int)X->seq_pages[b].size());
  }
  if (need > (int)X->free_pages.size())
    return fail(X, DF_ERR_CAPACITY, std::string(who) + ": page pool exhausted");
  EditQueue tq{X, X->Bf.kv_table};
  for (int b = 0; b < X->B; ++b)
    if (X->seq_len[b] >= 0) grow_slot(X, b, X->seq_len[b] + n, tq);
  tq.flush();
  return DF_OK;
}

void finish_steps(df_ctx* X, int n) {
  X->t += n;
  if (X->D.paged)
    for (int b = 0; b < X->B; ++b)
      if (X->seq_len[b] >= 0) X->seq_len[b] += n;
}

int count_kernel_nodes(cudaGraph_t g) {
  size_t n = 0;
  if (cudaGraphGetNodes(g, nullptr, &n) != cudaSuccess) return -1;
  std::vector<cudaGraphNode_t> nodes(n);
  if (cudaGraphGetNodes(g, nodes.data(), &n) != cudaSuccess) return -1;
  int k = 0;
  for (auto& nd : nodes) {
    cudaGraphNodeType t;
    if (cudaGraphNodeGetType(nd, &t) == cudaSuccess && t == cudaGraphNodeTypeKernel) ++k;
  }
  return k;
}

template <typename F>
df_status run_captured(df_ctx* X, GraphSlot& slot, const GraphKey& key, F&& enqueue, int repeat) {
  if (!X->use_graph) {
    for (int r = 0; r < repeat; ++r) enqueue();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(X, e, "kernel launch");
    X->last_kernels = -1;
    return DF_OK;
  }
  if (!slot.valid || !(slot.key == key)) {
    slot.reset();
    cudaGraph_t g = nullptr;
    cudaError_t e = cudaStreamBeginCapture(X->stream, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return cuda_fail(X, e, "cudaStreamBeginCapture");
    enqueue();
    cudaError_t le = cudaGetLastError();
    e = cudaStreamEndCapture(X->stream, &g);
    if (le != cudaSuccess) {
      if (g) cudaGraphDestroy(g);
      return cuda_fail(X, le, "kernel launch during capture");
    }
    if (e != cudaSuccess) return cuda_fail(X, e, "cudaStreamEndCapture");
    slot.kernels = count_kernel_nodes(g);
    e = cudaGraphInstantiate(&slot.exec, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) {
      slot.exec = nullptr;
      return cuda_fail(X, e, "cudaGraphInstantiate");
    }
    slot.key = key;
    slot.valid = true;
  }
  for (int r = 0; r < repeat; ++r) {
    cudaError_t e = cudaGraphLaunch(slot.exec, X->stream);
    if (e != cudaSuccess) return cuda_fail(X, e, "cudaGraphLaunch");
  }
  X->last_kernels = slot.kernels;
  return DF_OK;
}

// Prefill of n positions: all B sequences (nseq = B, slot0 = 0) or one slot
// (nseq = 1).  Positions must start at 0 (set by the caller).
df_status prefill_rows(df_ctx* X, const int32_t* tokens, int nseq, int n, int slot0, int B) {
  if (X->bp.enabled && X->tc.enabled && X->at.enabled && (!X->D.E || X->moe.enabled) && !X->force_generic) {
    // batched: every layer once per chunk of positions (kernels enqueued directly)
    df::bp_prefill(X->bp, X->tc, X->at, &X->moe, X->D, X->Bf, X->kv, X->emb1, X->attn_norm.data(),
                   X->mlp_norm.data(), X->router.data(), tokens, nseq, n, slot0, X->stream);
    df::launch_set_pos(X->Bf.ctrl, n, X->stream);
    if (X->D.paged) {
      EditQueue pq{X, X->Bf.kv_pos};
      for (int b = slot0; b < slot0 + nseq; ++b) pq.add(b, n);
      pq.flush();
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(X, e, "batched prefill launch");
    X->last_kernels = -1;
    return DF_OK;
  }
  // token-serial: one pass over all B primary rows per position; for one
  // slot the other rows compute at their own positions, where any value
  // written is rewritten by their next decode step before it is read
  GraphKey key{};
  key.p[0] = tokens;
  key.i[0] = n;
  key.i[1] = B;
  key.i[2] = X->force_generic;
  key.i[3] = nseq;
  key.i[4] = slot0;
  const int stride = nseq == 1 && B > 1 ? 0 : n;
  return run_captured(X, X->pre, key, [&] { enqueue_prefill_pos(X, tokens, stride, slot0, slot0 + nseq); }, n);
}

void setup_rope(df_ctx* X, std::vector<float>& host) {
  const Dims& D = X->D;
  int half = D.hd / 2;
  host.assign((size_t)(D.max_len + 1) * D.hd, 0.f);
  for (int t = 0; t <= D.max_len; ++t)
    for (int i = 0; i < half; ++i) {
      double ang = (double)t * std::pow((double)D.theta, -2.0 * i / D.hd);
      host[(size_t)t * D.hd + 2 * i] = (float)std::cos(ang);
      host[(size_t)t * D.hd + 2 * i + 1] = (float)std::sin(ang);
    }
}

}  // namespace

// ======================================================================== C ABI

extern "C" {

size_t df_workspace_bytes(const df_config* cfg, size_t* kv_bytes) {
  if (!valid_config(cfg, nullptr)) return 0;
  Dims D = make_dims(cfg);
  if (kv_bytes) *kv_bytes = kv_size(D);
  return layout(D, nullptr, nullptr);
}

df_status df_create(const df_config* cfg, const df_weights* w, void* kv_buf, void* workspace, void* cuda_stream,
                    df_ctx** out) {
  if (!out) return DF_ERR_ARG;
  *out = nullptr;
  std::string why;
  if (!valid_config(cfg, &why)) {
    fprintf(stderr, "df_create: %s\n", why.c_str());
    return DF_ERR_ARG;
  }
  if (!w || !kv_buf || !workspace) return DF_ERR_ARG;
  if (((uintptr_t)kv_buf & 255) || ((uintptr_t)workspace & 255)) return DF_ERR_ARG;
  int L = cfg->n_layers;
  if (!w->emb1 || !w->emb2 || !w->final_norm || !w->lm_head || !w->attn_norm || !w->wqkv || !w->wo ||
      !w->mlp_norm || !w->wgu || !w->wd || !w->a || !w->b || !w->c)
    return DF_ERR_ARG;
  if (cfg->n_experts && !w->router) return DF_ERR_ARG;
  for (int l = 0; l < L; ++l) {
    if (!w->attn_norm[l] || !w->wqkv[l] || !w->wo[l] || !w->mlp_norm[l] || !w->wgu[l] || !w->wd[l] || !w->a[l] ||
        !w->b[l] || !w->c[l])
      return DF_ERR_ARG;
    if (cfg->n_experts && !w->router[l]) return DF_ERR_ARG;
  }
  df_ctx* X = new df_ctx();
  X->cfg = *cfg;
  X->D = make_dims(cfg);
  X->emb1 = w->emb1;
  X->emb2 = w->emb2;
  X->final_norm = w->final_norm;
  X->lm_head = w->lm_head;
  X->attn_norm.assign(w->attn_norm, w->attn_norm + L);
  X->mlp_norm.assign(w->mlp_norm, w->mlp_norm + L);
  X->wqkv.assign(w->wqkv, w->wqkv + L);
  X->wo.assign(w->wo, w->wo + L);
  X->wgu.assign(w->wgu, w->wgu + L);
  X->wd.assign(w->wd, w->wd + L);
  X->a.assign(w->a, w->a + L);
  X->b.assign(w->b, w->b + L);
  X->c.assign(w->c, w->c + L);
  if (cfg->n_experts) X->router.assign(w->router, w->router + L);
  X->kv = kv_buf;
  X->ws = (char*)workspace;
  size_t ws_bytes = layout(X->D, &X->Bf, X->ws);
  if (cuda_stream) {
    X->stream = (cudaStream_t)cuda_stream;
  } else {
    cudaError_t e = cudaStreamCreate(&X->stream);  // blocking: ordered with the legacy stream
    if (e != cudaSuccess) {
      delete X;
      return DF_ERR_CUDA;
    }
    X->own_stream = true;
  }
  const char* ng = getenv("DF_NO_GRAPH");
  X->use_graph = !(ng && ng[0] == '1');
  const char* fg = getenv("DF_FORCE_GENERIC");
  X->force_generic = (fg && fg[0] == '1') ? 1 : 0;
  df::kernels_init();
  std::vector<float> rope;
  setup_rope(X, rope);
  X->seq_len.assign(X->D.maxB, -1);
  X->seq_pages.assign(X->D.maxB, {});
  std::vector<int> table;
  if (X->D.paged) {
    for (int p = X->D.NP - 2; p >= 0; --p) X->free_pages.push_back(p);  // page 0 is taken first
    table.assign((size_t)X->D.maxB * X->D.MPS, X->D.NP - 1);             // every entry at the sink
  }
  cudaError_t e = cudaMemsetAsync(X->ws, 0, ws_bytes, X->stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(X->Bf.rope, rope.data(), rope.size() * sizeof(float), cudaMemcpyHostToDevice, X->stream);
  if (e == cudaSuccess && !table.empty())
    e = cudaMemcpyAsync(X->Bf.kv_table, table.data(), table.size() * sizeof(int), cudaMemcpyHostToDevice,
                        X->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(X->stream);
  if (e != cudaSuccess) {
    fprintf(stderr, "df_create: %s\n", cudaGetErrorString(e));
    if (X->own_stream) cudaStreamDestroy(X->stream);
    delete X;
    return DF_ERR_CUDA;
  }
  std::string perr;
  if (!df::tc_plan_init(X->tc, X->D, X->Bf, X->wqkv, X->wo, X->wgu, X->wd, X->lm_head, &perr) ||
      (X->D.E && !df::moe_tc_init(X->moe, X->D, X->Bf, X->wgu, X->wd, &perr)) ||
      !df::attn_fast_init(X->at, X->D, X->kv, &perr) ||
      !df::mk_init(X->mk, X->D, X->Bf, X->Bf.mk, X->kv, X->wqkv, X->wo, X->wgu, X->wd, X->attn_norm, X->mlp_norm,
                   X->a, X->b, X->c, X->stream, &perr) ||
      !df::bp_init(X->bp, X->D, X->Bf.bp, &perr)) {
    fprintf(stderr, "df_create: %s\n", perr.c_str());
    if (X->own_stream) cudaStreamDestroy(X->stream);
    delete X;
    return DF_ERR_CUDA;
  }
  *out = X;
  return DF_OK;
}

static df_status set_batch(df_ctx* X, int B) {
  if (X->D.paged && B < X->B) {
    EditQueue tq{X, X->Bf.kv_table}, aq{X, X->Bf.kv_active}, pq{X, X->Bf.kv_pos};
    for (int b = B; b < X->B; ++b)
      if (X->seq_len[b] >= 0) {
        release_slot(X, b, tq);
        aq.add(b, 0);
        pq.add(b, 0);
      }
    tq.flush();
    aq.flush();
    pq.flush();
  }
  if (B != X->B) {
    X->dec.reset();
    X->dec_host[0].reset();
    X->dec_host[1].reset();
    X->pre.reset();
    X->dec_static.reset();
    X->gen.reset();
    X->B = B;
    X->splits = df::attn_splits(X->D, B);
    X->splits_fast = X->at.enabled ? df::attn_fast_splits(X->at, X->D, B) : X->splits;
    const char* pp = getenv("DF_PRINT_PLAN");
    if (pp && pp[0] == '1') {
      fprintf(stderr, "df plan: B=%d attention splits %d (CUDA-core path %d); clusters held at once by size:", B,
              X->splits_fast, X->splits);
      for (int sp = 1; sp <= 16; ++sp) fprintf(stderr, " %d:%d", sp, X->at.max_clusters[sp]);
      fprintf(stderr, "\n");
    }
    std::string perr;
    if (!df::tc_plan_batch(X->tc, X->D, B, &perr)) return fail(X, DF_ERR_CUDA, perr);
    if (!df::mk_batch(X->mk, X->D, X->Bf, B, &perr)) return fail(X, DF_ERR_CUDA, perr);
  }
  return DF_OK;
}

df_status df_prefill(df_ctx* X, const int32_t* tokens, int B, int n) {
  if (!X) return DF_ERR_ARG;
  if (B <= 0 || n < 0 || (n > 0 && !tokens)) return fail(X, DF_ERR_ARG, "df_prefill: bad arguments");
  if (B > X->cfg.max_batch) return fail(X, DF_ERR_CAPACITY, "df_prefill: B > max_batch");
  if (n > X->cfg.max_len) return fail(X, DF_ERR_CAPACITY, "df_prefill: n > max_len");
  if (X->D.paged && (size_t)B * pages_for(X->D, n) > (size_t)(X->D.NP - 1))
    return fail(X, DF_ERR_CAPACITY, "df_prefill: page pool too small for B sequences of n positions");
  df_status st = set_batch(X, B);
  if (st != DF_OK) return st;
  if (X->D.paged) {
    // every slot of the batch starts over: n positions, all active
    EditQueue tq{X, X->Bf.kv_table}, aq{X, X->Bf.kv_active}, pq{X, X->Bf.kv_pos};
    for (int b = 0; b < B; ++b)
      if (X->seq_len[b] >= 0) release_slot(X, b, tq);
    for (int b = 0; b < B; ++b) {
      grow_slot(X, b, n, tq);
      X->seq_len[b] = n;
      aq.add(b, 1);
      pq.add(b, 0);
    }
    tq.flush();
    aq.flush();
    pq.flush();
  }
  df::launch_set_pos(X->Bf.ctrl, 0, X->stream);
  X->t = 0;
  X->ready = true;
  if (n == 0) return DF_OK;
  st = prefill_rows(X, tokens, B, n, 0, B);
  if (st != DF_OK) return st;
  X->t = n;
  return DF_OK;
}



df_status df_set_length(df_ctx* X, int B, int t) {
  if (!X) return DF_ERR_ARG;
  if (B <= 0 || t < 0) return fail(X, DF_ERR_ARG, "df_set_length: bad arguments");
  if (B > X->cfg.max_batch) return fail(X, DF_ERR_CAPACITY, "df_set_length: B > max_batch");
  if (t > X->cfg.max_len) return fail(X, DF_ERR_CAPACITY, "df_set_length: t > max_len");
  if (X->D.paged && (size_t)B * pages_for(X->D, t) > (size_t)(X->D.NP - 1))
    return fail(X, DF_ERR_CAPACITY, "df_set_length: page pool too small");
  df_status st = set_batch(X, B);
  if (st != DF_OK) return st;
  if (X->D.paged) {
    EditQueue tq{X, X->Bf.kv_table}, aq{X, X->Bf.kv_active}, pq{X, X->Bf.kv_pos};
    for (int b = 0; b < B; ++b)
      if (X->seq_len[b] >= 0) release_slot(X, b, tq);
    for (int b = 0; b < B; ++b) {
      grow_slot(X, b, t, tq);
      X->seq_len[b] = t;
      aq.add(b, 1);
      pq.add(b, t);
    }
    tq.flush();
    aq.flush();
    pq.flush();
  }
  df::launch_set_pos(X->Bf.ctrl, t, X->stream);
  X->t = t;
  X->ready = true;
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DF_OK : cuda_fail(X, e, "df_set_length");
}

// One decode step replayed from the graph cached in `slot`.
static df_status decode_into(df_ctx* X, GraphSlot& slot, const int32_t* tokens, float* logp_mix, int32_t* argmax,
                             float* alpha) {
  df_status pst = prepare_steps(X, 1, "df_decode_step");
  if (pst != DF_OK) return pst;
  GraphKey key{};
  key.p[0] = tokens;
  key.p[1] = logp_mix;
  key.p[2] = argmax;
  key.p[3] = alpha;
  key.p[4] = X->dbg_logp1;
  key.p[5] = X->dbg_logp2;
  key.p[6] = X->dbg_topk;
  key.p[7] = X->dbg_router;
  key.i[0] = X->aux_on;
  key.i[1] = X->ungrouped;
  key.i[2] = X->B;
  key.i[3] = X->force_generic;
  StepOut o{logp_mix, argmax, alpha};
  df_status st = run_captured(X, slot, key, [&] { enqueue_decode(X, tokens, o); }, 1);
  if (st != DF_OK) return st;
  finish_steps(X, 1);
  return DF_OK;
}

df_status df_decode_step(df_ctx* X, const int32_t* tokens, float* logp_mix, int32_t* argmax, float* alpha) {
  if (!X) return DF_ERR_ARG;
  if (!tokens) return fail(X, DF_ERR_ARG, "df_decode_step: null tokens");
  if (!X->ready) return fail(X, DF_ERR_STATE, "df_decode_step before df_prefill");
  return decode_into(X, X->dec, tokens, logp_mix, argmax, alpha);
}

df_status df_generate(df_ctx* X, const int32_t* tokens, int n_steps, unsigned long long seed, int32_t* out_tokens,
                      float* logp_mix) {
  if (!X) return DF_ERR_ARG;
  if (n_steps < 0) return fail(X, DF_ERR_ARG, "df_generate: n_steps < 0");
  if (n_steps > 0 && (!tokens || !out_tokens)) return fail(X, DF_ERR_ARG, "df_generate: null tokens or out_tokens");
  if (!X->ready) return fail(X, DF_ERR_STATE, "df_generate before df_prefill");
  if (n_steps > X->cfg.max_len) return fail(X, DF_ERR_CAPACITY, "df_generate: n_steps > max_len");
  if (n_steps == 0) return DF_OK;
  df_status pst = prepare_steps(X, n_steps, "df_generate");
  if (pst != DF_OK) return pst;
  const int B = X->B;
  cudaError_t e = cudaSuccess;
  if (tokens != X->Bf.gen_tok)
    e = cudaMemcpyAsync(X->Bf.gen_tok, tokens, (size_t)B * 4, cudaMemcpyDeviceToDevice, X->stream);
  if (e != cudaSuccess) return cuda_fail(X, e, "df_generate: token copy");
  df::launch_set_seed(X->Bf.ctrl, seed, X->stream);
  GraphKey key{};
  key.p[0] = X->Bf.gen_tok;
  key.p[1] = logp_mix;
  key.p[4] = X->dbg_logp1;
  key.p[5] = X->dbg_logp2;
  key.p[6] = X->dbg_topk;
  key.p[7] = X->dbg_router;
  key.i[0] = X->aux_on;
  key.i[1] = X->ungrouped;
  key.i[2] = B;
  key.i[3] = X->force_generic;
  StepOut o{logp_mix, nullptr, nullptr, X->Bf.gen_tok, X->Bf.gen_hist};
  df_status st = run_captured(X, X->gen, key, [&] { enqueue_decode(X, X->Bf.gen_tok, o); }, n_steps);
  if (st != DF_OK) return st;
  finish_steps(X, n_steps);
  e = cudaMemcpy2DAsync(out_tokens, (size_t)B * 4, X->Bf.gen_hist, (size_t)X->D.maxB * 4, (size_t)B * 4, n_steps,
                        cudaMemcpyDeviceToDevice, X->stream);
  if (e != cudaSuccess) return cuda_fail(X, e, "df_generate: output copy");
  return DF_OK;
}

df_status df_sync(df_ctx* X) {
  if (!X) return DF_ERR_ARG;
  df::Ctrl h{};
  cudaError_t e = cudaMemcpyAsync(&h, X->Bf.ctrl, sizeof(h), cudaMemcpyDeviceToHost, X->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(X->stream);
  if (e != cudaSuccess) return cuda_fail(X, e, "df_sync");
  if (h.err) {
    char buf[256];
    if (h.err_info >= 300 && h.err_info < 400)  // persistent kernel: where it gave up
      snprintf(buf, sizeof(buf), "device error %d (detail %d: cta %d, awaited %d, target %d, seen %d, thread %d)",
               h.err, h.err_info, h.pad[0], h.pad[1], h.pad[2], h.pad[3], h.pad[4]);
    else
      snprintf(buf, sizeof(buf), "device error %d (detail %d)", h.err, h.err_info);
    X->err = buf;
    // the error is reported once; clear the latch so the context stays usable
    cudaMemsetAsync(&X->Bf.ctrl->err, 0, 2 * sizeof(int), X->stream);
    cudaStreamSynchronize(X->stream);
    return (df_status)h.err;
  }
  return DF_OK;
}

df_status df_decode_step_host(df_ctx* X, const int32_t* tokens, float* logp_mix, int32_t* argmax, float* alpha) {
  if (!X) return DF_ERR_ARG;
  if (!tokens) return fail(X, DF_ERR_ARG, "df_decode_step_host: null tokens");
  if (!X->ready) return fail(X, DF_ERR_STATE, "df_decode_step_host before df_prefill");
  df_status pst = prepare_steps(X, 1, "df_decode_step_host");  // capacity before any copy
  if (pst != DF_OK) return pst;
  int B = X->B, V = X->D.V;
  cudaError_t e = cudaSuccess;
  // staging area 0 may still be copied out by a pipelined step
  if (X->copy_done[0]) e = cudaStreamWaitEvent(X->stream, X->copy_done[0], 0);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(X->Bf.tokbuf, tokens, B * sizeof(int32_t), cudaMemcpyHostToDevice, X->stream);
  if (e != cudaSuccess) return cuda_fail(X, e, "token copy");
  df_status st = df_decode_step(X, X->Bf.tokbuf, logp_mix ? X->Bf.out_logp : nullptr, argmax ? X->Bf.out_arg : nullptr,
                                alpha ? X->Bf.out_alpha : nullptr);
  if (st != DF_OK) return st;
  if (logp_mix) e = cudaMemcpyAsync(logp_mix, X->Bf.out_logp, (size_t)B * V * 4, cudaMemcpyDeviceToHost, X->stream);
  if (e == cudaSuccess && argmax) e = cudaMemcpyAsync(argmax, X->Bf.out_arg, B * 4, cudaMemcpyDeviceToHost, X->stream);
  if (e == cudaSuccess && alpha) e = cudaMemcpyAsync(alpha, X->Bf.out_alpha, B * 4, cudaMemcpyDeviceToHost, X->stream);
  if (e != cudaSuccess) return cuda_fail(X, e, "output copy");
  return df_sync(X);
}

df_status df_decode_step_host_async(df_ctx* X, const int32_t* tokens, float* logp_mix, int32_t* argmax,
                                    float* alpha) {
  if (!X) return DF_ERR_ARG;
  if (!tokens) return fail(X, DF_ERR_ARG, "df_decode_step_host_async: null tokens");
  if (!X->ready) return fail(X, DF_ERR_STATE, "df_decode_step_host_async before df_prefill");
  df_status pst = prepare_steps(X, 1, "df_decode_step_host_async");  // capacity before any copy
  if (pst != DF_OK) return pst;
  cudaError_t e = cudaSuccess;
  if (!X->copy_stream) {
    e = cudaStreamCreateWithFlags(&X->copy_stream, cudaStreamNonBlocking);
    for (int k = 0; k < 2 && e == cudaSuccess; ++k) {
      e = cudaEventCreateWithFlags(&X->step_done[k], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&X->copy_done[k], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return cuda_fail(X, e, "df_decode_step_host_async: copy stream");
  }
  const int k = X->host_slot;
  const int B = X->B, V = X->D.V;
  float* dl = k ? X->Bf.out_logp2 : X->Bf.out_logp;
  int32_t* da = k ? X->Bf.out_arg2 : X->Bf.out_arg;
  float* dp = k ? X->Bf.out_alpha2 : X->Bf.out_alpha;
  // this staging area's previous contents must have left before the step
  // writes it again
  e = cudaStreamWaitEvent(X->stream, X->copy_done[k], 0);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(X->Bf.tokbuf, tokens, B * sizeof(int32_t), cudaMemcpyHostToDevice, X->stream);
  if (e != cudaSuccess) return cuda_fail(X, e, "df_decode_step_host_async: token copy");
  df_status st = decode_into(X, X->dec_host[k], X->Bf.tokbuf, logp_mix ? dl : nullptr, argmax ? da : nullptr,
                             alpha ? dp : nullptr);
  if (st != DF_OK) return st;
  e = cudaEventRecord(X->step_done[k], X->stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(X->copy_stream, X->step_done[k], 0);
  if (e == cudaSuccess && logp_mix)
    e = cudaMemcpyAsync(logp_mix, dl, (size_t)B * V * 4, cudaMemcpyDeviceToHost, X->copy_stream);
  if (e == cudaSuccess && argmax) e = cudaMemcpyAsync(argmax, da, B * 4, cudaMemcpyDeviceToHost, X->copy_stream);
  if (e == cudaSuccess && alpha) e = cudaMemcpyAsync(alpha, dp, B * 4, cudaMemcpyDeviceToHost, X->copy_stream);
  if (e == cudaSuccess) e = cudaEventRecord(X->copy_done[k], X->copy_stream);
  if (e != cudaSuccess) return cuda_fail(X, e, "df_decode_step_host_async: output copy");
  X->host_slot = k ^ 1;
  return DF_OK;
}

df_status df_host_wait(df_ctx* X) {
  if (!X) return DF_ERR_ARG;
  if (X->copy_stream) {
    cudaError_t e = cudaStreamSynchronize(X->copy_stream);
    if (e != cudaSuccess) return cuda_fail(X, e, "df_host_wait");
  }
  return df_sync(X);
}

df_status df_set_mode(df_ctx* X, int aux_on, int ungrouped) {
  if (!X) return DF_ERR_ARG;
  if ((aux_on != 0 && aux_on != 1) || (ungrouped != 0 && ungrouped != 1))
    return fail(X, DF_ERR_ARG, "df_set_mode: flags must be 0 or 1");
  X->aux_on = aux_on;
  X->ungrouped = ungrouped;
  return DF_OK;
}

df_status df_debug_outputs(df_ctx* X, float* logp1, float* logp2, int32_t* topk, float* router) {
  if (!X) return DF_ERR_ARG;
  if ((topk || router) && !X->cfg.n_experts) return fail(X, DF_ERR_ARG, "topk/router diagnostics need an MoE model");
  X->dbg_logp1 = logp1;
  X->dbg_logp2 = logp2;
  X->dbg_topk = topk;
  X->dbg_router = router;
  return DF_OK;
}

df_status df_time_op(df_ctx* X, int op, int iters, float* avg_ms) {
  if (!X || !avg_ms || iters <= 0) return DF_ERR_ARG;
  if (!X->ready) return fail(X, DF_ERR_STATE, "df_time_op before df_prefill");
  if (op < 0 || op > DF_OP_LAYERS) return fail(X, DF_ERR_ARG, "df_time_op: unknown op");
  if (op == DF_OP_MOE && !X->D.E) return fail(X, DF_ERR_ARG, "df_time_op: MoE op on a dense model");
  if ((op == DF_OP_GATEUP || op == DF_OP_DOWN) && X->D.E) return fail(X, DF_ERR_ARG, "df_time_op: dense op on MoE");
  int B = X->B;
  Rows R{B, 0, X->aux_on ? 2 * B : B};
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  cudaEventRecord(e0, X->stream);
  for (int i = 0; i < iters; ++i) {
    int l = i % X->D.L;
    Couple C = layer_couple(X, l, 0, 0);
    switch (op) {
      case DF_OP_QKV: op_qkv(X, l, R, C); break;
      case DF_OP_ATTN: op_attn(X, l, R); break;
      case DF_OP_WO: op_wo(X, l, R); break;
      case DF_OP_GATEUP: op_gateup(X, l, R, C); break;
      case DF_OP_DOWN: op_down(X, l, R, C); break;
      case DF_OP_LMHEAD: op_lm(X, R); break;
      case DF_OP_MOE: op_moe(X, l, R, C); break;
      case DF_OP_LAYERS: enqueue_layers(X, R, 0, 0); break;
    }
  }
  cudaEventRecord(e1, X->stream);
  cudaError_t e = cudaEventSynchronize(e1);
  float ms = 0.f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (e != cudaSuccess) return cuda_fail(X, e, "df_time_op");
  *avg_ms = ms / iters;
  return DF_OK;
}

int df_length(const df_ctx* X) {
  if (!X) return -1;
  if (!X->D.paged) return X->t;
  int m = 0;
  for (int b = 0; b < X->B; ++b) m = std::max(m, X->seq_len[b]);
  return m;
}

df_status df_set_batch(df_ctx* X, int B) {
  if (!X) return DF_ERR_ARG;
  if (!X->D.paged) return fail(X, DF_ERR_UNSUPPORTED, "df_set_batch: needs a paged cache (page_len > 0)");
  if (B <= 0 || B > X->cfg.max_batch) return fail(X, DF_ERR_ARG, "df_set_batch: B outside [1, max_batch]");
  df_status st = set_batch(X, B);
  if (st != DF_OK) return st;
  X->ready = true;
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DF_OK : cuda_fail(X, e, "df_set_batch");
}

df_status df_prefill_seq(df_ctx* X, int b, const int32_t* tokens, int n) {
  if (!X) return DF_ERR_ARG;
  if (!X->D.paged) return fail(X, DF_ERR_UNSUPPORTED, "df_prefill_seq: needs a paged cache (page_len > 0)");
  if (!X->ready || X->B <= 0) return fail(X, DF_ERR_STATE, "df_prefill_seq before df_set_batch or df_prefill");
  if (b < 0 || b >= X->B || n < 0 || (n > 0 && !tokens)) return fail(X, DF_ERR_ARG, "df_prefill_seq: bad arguments");
  if (n > X->cfg.max_len) return fail(X, DF_ERR_CAPACITY, "df_prefill_seq: n > max_len");
  EditQueue tq{X, X->Bf.kv_table}, aq{X, X->Bf.kv_active}, pq{X, X->Bf.kv_pos};
  const int had = (int)X->seq_pages[b].size();
  if (pages_for(X->D, n) > (int)X->free_pages.size() + had)
    return fail(X, DF_ERR_CAPACITY, "df_prefill_seq: page pool exhausted");
  if (X->seq_len[b] >= 0) release_slot(X, b, tq);
  grow_slot(X, b, n, tq);
  X->seq_len[b] = n;
  aq.add(b, 1);
  pq.add(b, 0);
  tq.flush();
  aq.flush();
  pq.flush();
  if (n > 0) {
    df::launch_set_pos(X->Bf.ctrl, 0, X->stream);
    df_status st = prefill_rows(X, tokens, 1, n, b, X->B);
    if (st != DF_OK) return st;
  }
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DF_OK : cuda_fail(X, e, "df_prefill_seq");
}

df_status df_release_seq(df_ctx* X, int b) {
  if (!X) return DF_ERR_ARG;
  if (!X->D.paged) return fail(X, DF_ERR_UNSUPPORTED, "df_release_seq: needs a paged cache (page_len > 0)");
  if (b < 0 || b >= X->cfg.max_batch) return fail(X, DF_ERR_ARG, "df_release_seq: bad slot");
  if (X->seq_len[b] < 0) return DF_OK;
  EditQueue tq{X, X->Bf.kv_table}, aq{X, X->Bf.kv_active}, pq{X, X->Bf.kv_pos};
  release_slot(X, b, tq);
  aq.add(b, 0);
  pq.add(b, 0);
  tq.flush();
  aq.flush();
  pq.flush();
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DF_OK : cuda_fail(X, e, "df_release_seq");
}

df_status df_seq_lengths(const df_ctx* X, int32_t* lengths) {
  if (!X || !lengths) return DF_ERR_ARG;
  for (int b = 0; b < X->cfg.max_batch; ++b) {
    if (X->D.paged)
      lengths[b] = b < X->B ? X->seq_len[b] : -1;
    else
      lengths[b] = (X->ready && b < X->B) ? X->t : -1;
  }
  return DF_OK;
}

int df_seq_pages(const df_ctx* X, int b, int32_t* pages, int cap) {
  if (!X || !X->D.paged || b < 0 || b >= X->cfg.max_batch) return -1;
  const auto& pg = X->seq_pages[b];
  for (int i = 0; i < (int)pg.size() && i < cap; ++i) pages[i] = pg[i];
  return (int)pg.size();
}

int df_step_kernels(const df_ctx* X) { return X ? X->last_kernels : -1; }

const char* df_last_error(const df_ctx* X) { return X ? X->err.c_str() : "null context"; }

void df_destroy(df_ctx* X) {
  if (!X) return;
  if (X->stream) cudaStreamSynchronize(X->stream);
  if (X->copy_stream) {
    cudaStreamSynchronize(X->copy_stream);
    cudaStreamDestroy(X->copy_stream);
  }
  for (int k = 0; k < 2; ++k) {
    if (X->step_done[k]) cudaEventDestroy(X->step_done[k]);
    if (X->copy_done[k]) cudaEventDestroy(X->copy_done[k]);
    X->dec_host[k].reset();
  }
  X->dec.reset();
  X->pre.reset();
  X->dec_static.reset();
  X->gen.reset();
  df::tc_plan_free(X->tc);
  df::moe_tc_free(X->moe);
  df::attn_fast_free(X->at);
  if (X->own_stream) cudaStreamDestroy(X->stream);
  delete X;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode step without workspace scratch for the split-attention partials.
//
// For callers that cannot allocate device memory at the point where they
// step the model: a serving loop that runs inside a fixed memory budget set
// at start-up, or code that assembles its own CUDA graph and may not add an
// allocation to it.  The partials that the split-KV attention kernels
// exchange (running max, running sum and unnormalised output per query row
// and split) live in the file-scope array below instead of the caller's
// workspace.  The array is reserved in every GPU's memory when the library is
// loaded and held until the process exits.
namespace {

constexpr size_t kStaticScratchFloats = size_t(1) << 20;  // 4 MiB of fp32
__device__ __align__(256) float g_step_scratch[kStaticScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_step_scratch on the current device.  In host code the
// symbol is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress.  It is looked up again on every call made outside
// stream capture (a device reset in between reloads the module at another
// address); a call made while `s` is being captured reuses the address
// found by the last call outside capture on that device.
cudaError_t static_scratch(cudaStream_t s, float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (cs == cudaStreamCaptureStatusNone || !g_scratch_ptr[dev]) {
    float* p = nullptr;
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_step_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

// Floats of the static array the step will use: the attention partials of
// the path the step takes.  The TMA attention kernel merges its KV splits
// in distributed shared memory and needs none; the persistent pass writes
// segment partials of its own layout; the CUDA-core attention writes one
// (head_dim + 2)-float partial per (sequence, KV head, split, query row).
size_t static_scratch_need(df_ctx* X, size_t* parts_out) {
  const Dims& D = X->D;
  const size_t parts = (size_t)X->B * D.Hkv * X->splits * 2 * D.G;
  *parts_out = parts;
  const int B = X->B;
  const bool two = X->aux_on && X->ungrouped;
  const Rows r0 = two ? Rows{B, 0, B} : Rows{B, 0, X->aux_on ? 2 * B : B};
  const Rows r1 = Rows{B, B, 2 * B};
  if (!X->force_generic && df::mk_can_run(X->mk, r0) && (!two || df::mk_can_run(X->mk, r1)))
    return df::mk_attn_partial_floats(D);
  if (!X->force_generic && df::attn_fast_can_run(X->at, D)) return 0;
  return parts * (D.hd + 2);
}

}  // namespace

extern "C" df_status df_decode_step_noalloc(df_ctx* X, const int32_t* tokens, float* logp_mix, int32_t* argmax,
                                            float* alpha) {
  if (!X) return DF_ERR_ARG;
  if (!tokens) return fail(X, DF_ERR_ARG, "df_decode_step_noalloc: null tokens");
  if (!X->ready) return fail(X, DF_ERR_STATE, "df_decode_step_noalloc before df_prefill");
  size_t parts = 0;
  const size_t need = static_scratch_need(X, &parts);
  if (need > kStaticScratchFloats) {
    char buf[160];
    snprintf(buf, sizeof(buf),
             "df_decode_step_noalloc: attention partials need %zu floats, the static scratch holds %zu", need,
             kStaticScratchFloats);
    return fail(X, DF_ERR_CAPACITY, buf);
  }
  float* scratch = nullptr;
  cudaError_t e = static_scratch(X->stream, &scratch);
  if (e != cudaSuccess) return cuda_fail(X, e, "cudaGetSymbolAddress");
  df_status pst = prepare_steps(X, 1, "df_decode_step_noalloc");
  if (pst != DF_OK) return pst;
  GraphKey key{};
  key.p[0] = tokens;
  key.p[1] = logp_mix;
  key.p[2] = argmax;
  key.p[3] = alpha;
  key.p[4] = X->dbg_logp1;
  key.p[5] = X->dbg_logp2;
  key.p[6] = X->dbg_topk;
  key.p[7] = scratch;
  key.i[0] = X->aux_on;
  key.i[1] = X->ungrouped;
  key.i[2] = X->B;
  key.i[3] = X->force_generic;
  key.i[4] = X->dbg_router != nullptr;
  StepOut o{logp_mix, argmax, alpha};
  // The step is enqueued with the partials pointed at the static array (the
  // split-attention partials of the kernel sequence, or those of the
  // persistent kernel, whichever path the step takes).
  Buffers saved = X->Bf;
  float* saved_apart = X->mk.apart;
  X->Bf.part_o = scratch;
  X->Bf.part_ml = scratch + parts * X->D.hd;
  X->mk.apart = scratch;
  df_status st = run_captured(X, X->dec_static, key, [&] { enqueue_decode(X, tokens, o); }, 1);
  X->Bf = saved;
  X->mk.apart = saved_apart;
  if (st != DF_OK) return st;
  finish_steps(X, 1);
  return DF_OK;
}
