/*
 * df.h — C ABI of the dual-flow Transformer decode library (libdf.so).
 *
 * The library runs the grouped dual-flow decode step on one GPU: the primary
 * flow (a standard causal Transformer that owns the only KV cache) and the
 * auxiliary flow (own token embedding, one-way coupling vectors a, b, c,
 * read-only on the primary cache) are stacked into one pass, so every weight
 * matrix and every KV region is read from HBM once per step for both flows.
 * Source: "Resumen Técnico: Dual-Flow Transformers" (gist.science technical
 * summary of arXiv 2608.12385), sections "Arquitectura Central",
 * "Mecanismos Clave" and "Costes de Inferencia vs. Entrenamiento".
 *
 * Conventions for every entry point
 *  - All pointers named "device" are CUDA device addresses owned by the
 *    caller; the library borrows them and never frees them.  They must stay
 *    valid until df_destroy.  "host" pointers are read or written before the
 *    call returns (df_decode_step_host) or copied during df_create.
 *  - Every call is asynchronous on the CUDA stream given to df_create unless
 *    stated otherwise.  Argument, capacity and state errors are detected on
 *    the host before anything is enqueued and leave the context unchanged.
 *  - Errors detected on the device (a bounded wait that ran out, an index out
 *    of range) are latched in a device word and reported by df_sync or by
 *    the next call.  No call exits or aborts the process.
 *  - df_last_error returns a NUL-terminated description of the last failure
 *    (owned by the context, valid until the next call on it).
 *
 * Matrices are row-major [rows][cols] (PyTorch nn.Linear layout: out x in).
 * Element type of matrices, embeddings and the KV cache is cfg.dtype (fp32
 * or bf16); norm gains and coupling vectors are always fp32.
 */
#ifndef DF_H
#define DF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DF_OK = 0,
  DF_ERR_ARG = 1,          /* null pointer, bad size, unsupported combination      */
  DF_ERR_CUDA = 2,         /* a CUDA runtime/driver call failed                   */
  DF_ERR_CAPACITY = 3,     /* batch > max_batch or position >= max_len            */
  DF_ERR_STATE = 4,        /* decode before prefill, etc.                         */
  DF_ERR_TIMEOUT = 5,      /* a bounded device wait ran out (device error word)   */
  DF_ERR_UNSUPPORTED = 6,  /* shape the kernels do not implement                  */
  DF_ERR_DEVICE = 7        /* device-side bounds check failed (token id, expert)  */
} df_status;

typedef enum { DF_F32 = 0, DF_BF16 = 1 } df_dtype;

/* Model shape and capacity.  n_experts == 0 selects the dense SwiGLU MLP of
 * width ffn_hidden; n_experts > 0 selects the MoE MLP with top_k experts of
 * width expert_hidden ("Mecanismos Clave", Replay de Router). */
typedef struct {
  int n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_hidden, vocab;
  int n_experts, top_k, expert_hidden;
  float rope_theta, norm_eps;
  int dtype;               /* df_dtype */
  int max_batch, max_len;  /* capacity of the KV cache and workspace        */
  int aux_top_k;           /* MoE: experts per token of the auxiliary flow:
                              the primary's top_k (replayed) plus
                              aux_top_k - top_k chosen from its own router
                              logits among the other experts (0 = top_k).
                              Prefill cost is unchanged; decode reads the
                              extra experts' weights once for the batch.   */
  int page_len;            /* 0: contiguous KV cache, every sequence of the
                              batch at one common position.  A power of two
                              >= 64: paged KV cache with per-sequence
                              lengths (ragged batches, slots filled and
                              released between steps; see df_prefill_seq).  */
  int n_pages;             /* paged mode: pages of page_len positions in the
                              pool shared by all sequences (>= 1)           */
} df_config;

/* Parameter set (all device pointers; the struct and its per-layer arrays
 * are host memory copied by df_create).  Both flows share every matrix
 * except the token embeddings ("Arquitectura Central", Compartición de Pesos
 * and Separación).
 *
 *  emb1, emb2   [vocab][d]                primary / auxiliary token embeddings
 *  final_norm   [d] fp32                  final RMSNorm gain (shared)
 *  lm_head      [vocab][d]                output matrix (shared, untied)
 *  attn_norm[l] [d] fp32
 *  wqkv[l]      [(Hq + 2*Hkv)*hd][d]      rows: Wq, then Wk, then Wv
 *  wo[l]        [d][Hq*hd]
 *  mlp_norm[l]  [d] fp32
 *  wgu[l]       dense: [2F][d]; MoE: [E][2Fe][d].  Gate and up rows are
 *               interleaved in blocks of 64: rows 128j..128j+63 are gate rows
 *               64j..64j+63 and rows 128j+64..128j+127 the matching up rows.
 *  wd[l]        dense: [d][F]; MoE: [E][d][Fe]
 *  router[l]    MoE: [E][d]; NULL for dense models
 *  a[l]         [Hq*hd] fp32   query coupling:        Q2 = Wq·u2 + a ⊙ q1 (pre-RoPE)
 *  b[l]         [F or Fe] fp32 MLP-intermediate coupling: z2 += b ⊙ z1
 *  c[l]         [d] fp32       MLP-output coupling:   y2 += c ⊙ y1
 */
typedef struct {
  const void* emb1;
  const void* emb2;
  const float* final_norm;
  const void* lm_head;
  const float* const* attn_norm;
  const void* const* wqkv;
  const void* const* wo;
  const float* const* mlp_norm;
  const void* const* wgu;
  const void* const* wd;
  const void* const* router;
  const float* const* a;
  const float* const* b;
  const float* const* c;
} df_weights;

typedef struct df_ctx df_ctx;

/* Sizes of the two device buffers the caller allocates for a configuration:
 * returns the workspace size in bytes and stores the KV-cache size in
 * *kv_bytes (if non-NULL).  Returns 0 for an invalid configuration.
 *
 * KV-cache layout (primary flow only; the auxiliary flow never writes it):
 *   [n_layers][2 (K, V)][max_batch][n_kv_heads][max_len][head_dim] of dtype,
 * K stored after RoPE.  Positions 0..t-1 of sequence b are valid after
 * prefill or decode has reached position t. */
size_t df_workspace_bytes(const df_config* cfg, size_t* kv_bytes);

/* Create a context.  kv_buf and workspace are device buffers of the sizes
 * df_workspace_bytes reported (256-byte aligned); cuda_stream is a
 * cudaStream_t (NULL = legacy default stream).  Builds TMA descriptors and
 * launch plans; enqueues only memsets. */
df_status df_create(const df_config* cfg, const df_weights* w, void* kv_buf, void* workspace,
                    void* cuda_stream, df_ctx** out);

/* Prefill: run the primary flow alone over positions 0..n-1 of B sequences
 * and write their K/V ("Arquitectura Central": the auxiliary flow is
 * skipped during prefill).  tokens: device int32 [B][n].  Resets the
 * position to n.  For a prompt of length P the caller prefills P-1 tokens
 * and passes the last prompt token to the first df_decode_step, where the
 * auxiliary flow is active.  n may be 0 (empty prompt). */
df_status df_prefill(df_ctx* ctx, const int32_t* tokens, int B, int n);

/* Declare that the caller has written positions 0..t-1 of B sequences into
 * the KV cache itself (restoring a saved cache).  Next decode runs at t. */
df_status df_set_length(df_ctx* ctx, int B, int t);

/* One grouped decode step at position t for the B sequences of the last
 * prefill: both flows, K/V appended at t for the primary flow only, then the
 * mixture p_mix = alpha*p1 + (1-alpha)*p2 with alpha = 0.5 + 0.5*sum(p1^2)
 * ("Mecanismos Clave", Objetivo de Mezcla).  tokens: device int32 [B].
 * Outputs (device, each may be NULL): logp_mix fp32 [B][vocab],
 * argmax int32 [B] (lowest index among equal maxima), alpha fp32 [B].
 * Advances the position to t+1.  DF_ERR_CAPACITY if t >= max_len. */
df_status df_decode_step(df_ctx* ctx, const int32_t* tokens, float* logp_mix, int32_t* argmax,
                         float* alpha);

/* The same step with HOST buffers: copies tokens (host int32 [B]) to the
 * device, runs the step, copies the outputs back (host, each may be NULL)
 * and synchronises the stream before returning.  Pinned host memory gives
 * asynchronous copies; pageable memory works but is slower. */
df_status df_decode_step_host(df_ctx* ctx, const int32_t* tokens, float* logp_mix,
                              int32_t* argmax, float* alpha);

/* Pipelined form of df_decode_step_host for callers whose next tokens do not
 * depend on this step's outputs (teacher forcing, scoring): enqueues the
 * copy of tokens (host int32 [B]) to the device, the step, and the copies of
 * the outputs (host, each may be NULL) back to the host, and returns without
 * waiting.  The output copies run on a second stream of the context from one
 * of two device staging areas used in turn, so they overlap the next step's
 * kernels.  The host buffers belong to the library until df_host_wait
 * returns: tokens must not change and the outputs are not valid before
 * then.  Errors of the enqueue are returned at once; device-detected errors
 * by df_host_wait. */
df_status df_decode_step_host_async(df_ctx* ctx, const int32_t* tokens, float* logp_mix,
                                    int32_t* argmax, float* alpha);

/* Waits until every step enqueued by df_decode_step_host_async has
 * completed and its outputs are in host memory, then reports like df_sync. */
df_status df_host_wait(df_ctx* ctx);

/* Generation: n_steps decode steps on the device, each fed the token drawn
 * from p_mix at the step before ("Problema Central": decode generates tokens
 * one at a time; "Mecanismos Clave", Objetivo de Mezcla: p_mix is the
 * next-token distribution).  The first step is fed tokens (device int32
 * [B]); the step at position t draws, for sequence b,
 *     x = argmax_v ( log p_mix[v] + g_v ),  g_v = -log(-log u_v)
 * (Gumbel-max: one draw from p_mix itself, no temperature or truncation;
 * lowest index among equal maxima), with u_v = (2*(w >> 41) + 1) / 2^24 and
 * w word (v mod 4) of Philox4x64-10 (Salmon et al., SC 2011) at counter
 * (v div 4, b, t, 0) and key (seed, 0).  A draw therefore depends only on
 * (seed, t, b, p_mix).
 * Outputs (device): out_tokens int32 [n_steps][B], the token drawn at each
 * step (row s is the input of step s+1); logp_mix fp32 [B][vocab] or NULL,
 * the last step's log p_mix.  The debug outputs and the mode (aux_on,
 * ungrouped) apply as for df_decode_step; with aux_on = 0 the draw is from
 * p1.  Advances the position by n_steps.  DF_ERR_CAPACITY (nothing enqueued)
 * if t + n_steps > max_len; n_steps = 0 does nothing.  tokens may alias
 * out_tokens of an earlier call (it is copied before the first step). */
df_status df_generate(df_ctx* ctx, const int32_t* tokens, int n_steps, unsigned long long seed,
                      int32_t* out_tokens, float* logp_mix);

/* Execution mode for later decode steps.
 *  aux_on = 0: standard decode (primary flow only); logp_mix receives
 *              log p1, alpha receives 1.
 *  ungrouped = 1: the ablation that runs the primary flow and then the
 *              auxiliary flow as two passes, re-reading every weight and KV
 *              region; results are identical to the grouped step. */
df_status df_set_mode(df_ctx* ctx, int aux_on, int ungrouped);

/* Optional per-step diagnostics written by later decode steps (device
 * pointers, each may be NULL): logp1, logp2 fp32 [B][vocab]; topk int32
 * [n_layers][B][k] with k = max(top_k, aux_top_k): entries 0..top_k-1 are
 * the primary experts (descending router logit), entries top_k..k-1 the
 * auxiliary flow's own experts (descending auxiliary router logit; written
 * only while the auxiliary flow runs); router fp32 [n_layers][B][n_experts]
 * (primary router logits). */
df_status df_debug_outputs(df_ctx* ctx, float* logp1, float* logp2, int32_t* topk, float* router);

/* Decode step without workspace scratch for the attention partials.
 *
 * The method described by the paper has no counterpart to this entry point:
 * it exists for callers that cannot allocate device memory where they step
 * the model (a serving loop held to a fixed memory budget after start-up,
 * or code that assembles its own CUDA graph and may not add an allocation
 * to it).  Same arguments, outputs and position handling as df_decode_step.
 * The partials that the split-KV attention kernels exchange are kept in a
 * file-scope device array of 2^20 floats (4 MiB) that every GPU loading the
 * library reserves until the process exits; the workspace given to
 * df_create is still used for everything else.  Which partials the step
 * writes depends on the attention path it takes: the TMA attention kernel
 * (bf16, head_dim 128) merges its KV splits in distributed shared memory and
 * writes none; the CUDA-core attention writes B * n_kv_heads * splits *
 * 2 * (n_heads/n_kv_heads) rows of head_dim + 2 floats; the persistent pass
 * (DF_MK=1) writes up to min(max_batch, 16) * n_kv_heads * 16 segments of
 * 8 * (head_dim + 2) floats.
 *  - Returns DF_ERR_CAPACITY before enqueuing anything when the partials of
 *    the path the current batch takes exceed the array.
 *  - The array's device address is looked up (cudaGetSymbolAddress) on every
 *    call made outside stream capture, and reused from the last such call
 *    during capture: make the first call on a device before any capture.
 *  - All calls in the process share the one array and it keeps the last
 *    call's contents (every slot a call reads is written by that call first);
 *    calls that overlap on the GPU, from any context or stream, race. */
df_status df_decode_step_noalloc(df_ctx* ctx, const int32_t* tokens, float* logp_mix, int32_t* argmax,
                                 float* alpha);

/* ---- Paged KV cache: ragged batches and continuous decode -------------
 *
 * With page_len > 0 the cache is a pool of n_pages pages, each holding
 * page_len positions of one sequence for every layer and KV head
 * ([n_layers][2][n_pages + 1][n_kv_heads][page_len][head_dim]; the last page
 * is a sink that free slots write into).  Every sequence (slot b of the
 * batch) has its own length: a decode step processes each active slot at its
 * own position t_b (RoPE angle, cache slot and attention range 0..t_b; the
 * draw of df_generate uses t_b too), so the result for a slot is the one a
 * batch of that sequence alone would give ("Arquitectura Central": one
 * persistent primary cache per sequence; the auxiliary flow reads it at the
 * same position).  Pages are taken from the pool when a slot's next position
 * starts a page and returned when the slot is released or prefilled again.
 * df_prefill and df_set_length prefill / declare all B slots with one length;
 * the calls below manage single slots.  Steps decode the slots [0, B) of the
 * last df_set_batch / df_prefill / df_set_length: free slots are computed
 * too, their outputs are unspecified and nothing of theirs is kept.  A step
 * returns DF_ERR_CAPACITY, with nothing enqueued, when an active slot would
 * pass max_len or the pool has no page for a position it must write. */

/* Paged mode: decode B slots per step from now on; slots >= B are released,
 * slots < B keep their sequences.  DF_ERR_UNSUPPORTED in contiguous mode. */
df_status df_set_batch(df_ctx* ctx, int B);

/* Paged mode: prefill slot b (0 <= b < B) with its own prompt of n
 * positions (tokens: device int32 [n]), primary flow only; the slot's old
 * sequence, if any, is released first.  The next decode step processes the
 * slot at position n.  Other slots are unchanged.  DF_ERR_CAPACITY (slot
 * left as it was) when the pool cannot hold n positions. */
df_status df_prefill_seq(df_ctx* ctx, int b, const int32_t* tokens, int n);

/* Paged mode: release slot b, returning its pages to the pool. */
df_status df_release_seq(df_ctx* ctx, int b);

/* Length of every slot (host int32 [max_batch]): -1 for free slots and slots
 * >= B.  Contiguous mode: the common length for b < B. */
df_status df_seq_lengths(const df_ctx* ctx, int32_t* lengths);

/* Paged mode: the physical pages of slot b in logical order (host int32,
 * up to cap written); returns the slot's page count, -1 on a bad argument
 * or in contiguous mode. */
int df_seq_pages(const df_ctx* ctx, int b, int32_t* pages, int cap);

/* Synchronise the stream and report any latched device error. */
df_status df_sync(df_ctx* ctx);

/* Current position (number of valid cache positions); paged mode: the
 * largest length among the active slots. */
int df_length(const df_ctx* ctx);

/* Number of kernels in the last captured step graph (decode or prefill
 * position), or -1 when steps run without graph capture. */
int df_step_kernels(const df_ctx* ctx);

/* Bench hook: re-run one operation of the step `iters` times on the
 * context's stream, cycling through the layers (so consecutive launches read
 * different weights and no launch is served from L2 by its predecessor),
 * bracketed by CUDA events; *avg_ms receives the mean time per launch.
 * Operations re-execute on the current buffers and are idempotent for the
 * cache contents of valid positions.  Needs a previous decode step. */
enum {
  DF_OP_QKV = 0,     /* fused QKV projection + coupling + RoPE + cache append */
  DF_OP_ATTN = 1,    /* shared-KV split attention + split merge               */
  DF_OP_WO = 2,      /* output projection + residual                         */
  DF_OP_GATEUP = 3,  /* gate/up projection + SwiGLU + b coupling (dense)     */
  DF_OP_DOWN = 4,    /* down projection + c coupling + residual (dense)      */
  DF_OP_LMHEAD = 5,  /* LM head                                              */
  DF_OP_MOE = 6,     /* router + replayed experts + combine (MoE)            */
  DF_OP_LAYERS = 7   /* every layer of a grouped pass: the per-layer kernel
                        sequence, or one persistent-kernel launch where that
                        is enabled (DF_MK=1) and applies (dense bf16,
                        head_dim 128, at most 32 stacked rows); iterations
                        are whole passes, not layers                        */
};
df_status df_time_op(df_ctx* ctx, int op, int iters, float* avg_ms);

const char* df_last_error(const df_ctx* ctx);

/* Release host state (graphs, plans).  Device buffers stay with the caller. */
void df_destroy(df_ctx* ctx);

#ifdef __cplusplus
}
#endif

#endif /* DF_H */
