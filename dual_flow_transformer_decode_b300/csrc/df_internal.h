// Internal interface between the C-ABI runtime (df_runtime.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "common.cuh"

namespace df {

// Programmatic dependent launch (on unless DF_NO_PDL=1): a kernel may start
// while its predecessor drains; every kernel calls griddepcontrol.wait before
// it touches the predecessor's outputs.
bool pdl_enabled();

template <typename... KArgs, typename... Args>
inline void launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t lc{};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  lc.attrs = at;
  lc.numAttrs = 1;
  cudaLaunchKernelEx(&lc, kernel, std::forward<Args>(args)...);
}

// Model dimensions plus derived sizes, fixed at df_create.
struct Dims {
  int L, d, Hq, Hkv, hd, F, V, E, k, Fe;
  int ka;          // MoE experts per auxiliary token (>= k; k + auxiliary fan-out)
  float theta, eps;
  int bf16;        // 1: bf16 storage, 0: fp32
  int maxB, max_len;
  int qdim, kvdim, qkvn, G, Fm;   // Fm = MLP hidden of one expert or of the dense MLP
  int esz;         // element size of dtype
  int sms;         // streaming multiprocessors of the device
  // KV-cache pages (see KvMap): contiguous mode NP = maxB, PG = max_len,
  // MPS = 1; paged mode NP = pool pages + 1 (the last is a sink written by
  // free slots), PG a power of two >= 64, MPS = ceil(max_len / PG)
  int paged, NP, PG, MPS, pg_shift;
  size_t kv_layer_elems() const { return (size_t)2 * NP * Hkv * PG * hd; }  // one layer's K and V blocks
  size_t kv_half_elems() const { return (size_t)NP * Hkv * PG * hd; }       // the K (or V) block of a layer
};

// Device buffers carved out of the caller's workspace.
struct Buffers {
  Ctrl* ctrl;
  KvMap kvm;        // cache addressing (page table, positions, active flags in paged mode)
  int* kv_table;    // paged mode: [maxB][MPS] page table
  int* kv_pos;      // paged mode: [maxB] positions
  int* kv_active;   // paged mode: [maxB] active flags
  int* tokbuf;      // [maxB]   tokens of a host-buffer step
  float* h;         // [2maxB][d] fp32 residual rows (0..B-1 primary, B..2B-1 auxiliary)
  void* u;          // [Mpad][d]  normed rows (GEMM input, dtype)
  float* un;        // [2maxB][d] normed rows, unrounded (router input)
  float* qatt;      // [2maxB][qdim] rotated, quantised queries
  void* o;          // [Mpad][qdim] attention output (GEMM input, dtype)
  void* z;          // [Mpad][F]  SwiGLU output (GEMM input, dtype)
  float* raw;       // [Mpad][rawN] fp32 GEMM output before the epilogue (CUDA-core path)
  int rawN;
  float* logits;    // [2maxB][V]
  float* gpart;     // tensor-core GEMM split-K partial tiles reduced through L2 (tc_partial_floats)
  float* part_o;    // attention split partials: [parts][hd]
  float* part_ml;   // [parts][2] (running max, running sum)
  size_t parts_cap; // number of (b, kv head, split, row) partial slots
  float* q1s;       // [L][maxB][qdim] saved primary pre-RoPE queries (ungrouped)
  float* z1s;       // [L][maxB][F] (MoE: [L][maxB][k][Fe]) saved primary MLP hidden
  float* y1s;       // [L][maxB][d] saved primary MLP output
  int* topk;        // [L][maxB][k] primary expert sets
  float* gate;      // [2maxB][ka] gate weights per row (primary rows use the first k)
  int* topkx;       // [maxB][ka-k] this layer's auxiliary-own experts
  int* ecount;      // [E]
  int* elist;       // [E][maxB] entries: b*k + j (replayed), B*k + b*(ka-k) + j (auxiliary-own)
  void* zE;         // [2][maxB][ka][Fe] expert hidden (dtype)
  float* yE;        // [2][maxB][ka][d] expert outputs fp32
  int* eslot;       // [maxB*ka] position of each entry in its expert's list
  int* ticket;      // [1] arrivals at the routing launch (the last CTA builds the entry lists and resets it)
  void* xg;         // [E][nxe][d] packed expert input rows (tensor-core MoE path)
  void* zEt;        // [E][nxe][Fe] packed expert hidden rows
  float* yEt;       // [E][nxe][d] packed expert outputs
  float* out_logp;  // [maxB][V] host-step staging
  int* out_arg;     // [maxB]
  float* out_alpha; // [maxB]
  float* out_logp2; // second staging area of the pipelined host step
  int* out_arg2;
  float* out_alpha2;
  int* gen_tok;     // [maxB] generation: the next step's input tokens (written by the draw)
  int* gen_hist;    // [max_len][maxB] generation: the token drawn at each position
  float* rope;      // [max_len][hd/2][2] cos, sin
  void* mk;         // persistent-kernel region (maps, task lists, counters, partials)
  size_t mk_bytes;
  void* bp;         // batched-prefill chunk buffers
  size_t bp_bytes;
};

// Which rows of the stacked block a launch works on.
struct Rows {
  int B;        // batch
  int lo, hi;   // active stacked rows [lo, hi): [0,B) primary, [B,2B) auxiliary, [0,2B) both
  bool has_primary() const { return lo < B; }
  bool has_aux() const { return hi > B; }
};

// Coupling sources for the auxiliary rows of one layer.
//  grouped   (saved == 0): the primary values come from the same launch (rows 0..B-1)
//  ungrouped (saved == 1): they come from the q1s / z1s / y1s buffers of layer l
struct Couple {
  int saved;    // read partners from the saved buffers
  int save;     // write primary values to the saved buffers
  float* q1s;   // layer slice
  float* z1s;
  float* y1s;
};

// ------------------------------------------------------------ basic kernels
void kernels_init();   // one-time function attributes (dynamic shared memory limits)
void launch_set_pos(Ctrl* c, int t, cudaStream_t s);
// End of a pass: step counter + 1; paged mode: positions of the active
// sequences in [lo, hi) + 1.
void launch_advance_pos(const Buffers& Bf, int lo, int hi, cudaStream_t s);
// Up to kIntEdits writes dst[idx[i]] = val[i], in order, on the stream.
constexpr int kIntEdits = 48;
struct IntEdits {
  int n;
  int idx[kIntEdits];
  int val[kIntEdits];
};
void launch_int_edits(int* dst, const IntEdits& e, cudaStream_t s);
void launch_set_seed(Ctrl* c, unsigned long long seed, cudaStream_t s);
void launch_embed(const Dims& D, const Buffers& Bf, const void* emb1, const void* emb2,
                  const int32_t* tokens, int tok_stride, int use_pos, const Rows& R, cudaStream_t s);
void launch_rmsnorm(const Dims& D, const Buffers& Bf, const float* g, void* out, float* out_f32,
                    const Rows& R, cudaStream_t s);
// RMSNorm of rows 0..rows-1 of h (row stride d) into out (storage type).
void launch_rmsnorm_rows(const Dims& D, const float* h, const float* g, void* out, int rows, cudaStream_t s,
                         float* out_f32 = nullptr);
// Router logits rlog[m][E] of rows 0..rows-1 of an unrounded normed buffer.
void launch_router_rows(const Dims& D, const void* Wr, const float* un, float* rlog, int rows, cudaStream_t s);

// CUDA-core GEMV: out[m][n] = sum_k W[n][k] X[m][k] for rows m in [lo, hi)
// (W and X in the model's storage type).
void launch_gemv(const Dims& D, const void* W, int N, int K, const void* X, int ldx, float* out, int ldo,
                 const Rows& R, cudaStream_t s);

// Epilogues over the fp32 GEMM output `raw`.
void launch_ep_qkv(const Dims& D, const Buffers& Bf, const float* raw, int ldr, const float* a,
                   void* kv, int layer, const Couple& C, const Rows& R, cudaStream_t s);
void launch_ep_swiglu(const Dims& D, const Buffers& Bf, const float* raw, int ldr, const float* bvec,
                      const Couple& C, const Rows& R, cudaStream_t s);
void launch_ep_down(const Dims& D, const Buffers& Bf, const float* raw, int ldr, const float* cvec,
                    const Couple& C, const Rows& R, cudaStream_t s);
void launch_ep_residual(const Dims& D, const Buffers& Bf, const float* raw, int ldr, const Rows& R,
                        cudaStream_t s);

// Attention (split-KV) and the merge of split partials into o.
int attn_splits(const Dims& D, int B);
void launch_attention_generic(const Dims& D, const Buffers& Bf, const void* kv, int layer, int splits,
                              const Rows& R, cudaStream_t s);
void launch_attn_combine(const Dims& D, const Buffers& Bf, int splits, const Rows& R, cudaStream_t s);

// Softmax / mixture / argmax.
// Softmax of both flows, mixture, log p_mix and its argmax; with sample_tok
// set, also one draw from p_mix per sequence (written to sample_tok[b] and,
// if set, to sample_hist[t][b], row stride maxB).
void launch_mix(const Dims& D, const Buffers& Bf, int B, int aux_on, float* logp_mix, int32_t* argmax,
                float* alpha, float* logp1, float* logp2, int32_t* sample_tok, int32_t* sample_hist,
                cudaStream_t s);

// MoE with router replay.
// Router logits of rows R and routing (top-k of the primary rows when
// `select`, else the saved choice; gates of both flows; per-expert entry
// lists) in one launch.
void launch_router_route(const Dims& D, const Buffers& Bf, const void* Wr, int layer, int select, const Rows& R,
                         int32_t* dbg_topk, float* dbg_router, cudaStream_t s);
void launch_moe_gateup_generic(const Dims& D, const Buffers& Bf, const void* wgu, const float* bvec,
                               const Couple& C, const Rows& R, cudaStream_t s);
void launch_moe_down_generic(const Dims& D, const Buffers& Bf, const void* wd, const Rows& R,
                             cudaStream_t s);
void launch_moe_combine(const Dims& D, const Buffers& Bf, const float* cvec, const Couple& C,
                        const Rows& R, cudaStream_t s);

}  // namespace df
