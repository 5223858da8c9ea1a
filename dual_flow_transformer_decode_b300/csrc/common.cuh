// Shared device helpers for the dual-flow decode kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace df {

// Device error codes latched in the control block (values match df_status).
enum : int { kErrNone = 0, kErrTimeout = 5, kErrDevice = 7 };

// Control block at the start of the workspace.
struct Ctrl {
  int t;          // current position (number of valid cache positions)
  int err;        // first latched device error (0 = none)
  int err_info;   // kernel-specific detail for the first error
  int mk_abort;   // set by a persistent-kernel CTA that gave up; the others stop waiting
  unsigned long long seed;  // key of the sampling noise (generation)
  int gen_row;    // generation: history row of the current step (reset with the seed)
  int pad[57];
};
static_assert(sizeof(Ctrl) == 256, "control block layout");

__device__ __forceinline__ void latch_error(Ctrl* c, int code, int info) {
  if (atomicCAS(&c->err, 0, code) == 0) c->err_info = info;
}

// KV-cache addressing.  The cache is [L][2][NP][Hkv][PG][hd]: per layer a K
// block then a V block, each made of NP pages of PG positions per KV head.
// Paged mode: position p of sequence b lives in page
// table[b*MPS + (p >> pg_shift)] at offset p & (PG - 1), and each sequence
// has its own position pos[b].  Contiguous mode (table == nullptr): one page
// of max_len positions per sequence (page b, offset p) and every sequence at
// position ctrl->t.
struct KvMap {
  const int* table;  // [maxB][MPS] physical page of each logical page, or nullptr
  const int* pos;    // [maxB] current position of each sequence (paged mode)
  const int* active; // [maxB] 1 for sequences that advance (paged mode)
  int NP, PG, MPS, pg_shift;
};

__device__ __forceinline__ int kv_seq_pos(const KvMap& m, const Ctrl* c, int b) {
  return m.table ? m.pos[b] : c->t;
}
__device__ __forceinline__ int kv_page(const KvMap& m, int b, int p) {
  return m.table ? m.table[b * m.MPS + (p >> m.pg_shift)] : b;
}
__device__ __forceinline__ int kv_off(const KvMap& m, int p) { return m.table ? (p & (m.PG - 1)) : p; }
// Element index of (layer, kv = 0 for K / 1 for V, page, KV head g, offset).
__device__ __forceinline__ size_t kv_index(const KvMap& m, int Hkv, int hd, int layer, int kv, int page, int g,
                                           int off) {
  return ((((size_t)(layer * 2 + kv) * m.NP + page) * Hkv + g) * m.PG + off) * hd;
}

// Philox4x64 with 10 rounds (Salmon, Moraes, Dror and Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC 2011): a keyed bijection of a 256-bit
// counter.  Each round multiplies counter words 0 and 2 by two fixed odd
// constants and mixes each product's high half into the other two words and
// the key; the key advances by two Weyl increments between rounds.
struct Philox4x64Out {
  unsigned long long w[4];
};
__device__ __forceinline__ Philox4x64Out philox4x64_10(unsigned long long c0, unsigned long long c1,
                                                       unsigned long long c2, unsigned long long c3,
                                                       unsigned long long k0, unsigned long long k1) {
  constexpr unsigned long long kM0 = 0xD2E7470EE14C6C93ull, kM1 = 0xCA5A826395121157ull;
  constexpr unsigned long long kW0 = 0x9E3779B97F4A7C15ull, kW1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const unsigned long long lo0 = kM0 * c0, hi0 = __umul64hi(kM0, c0);
    const unsigned long long lo1 = kM1 * c2, hi1 = __umul64hi(kM1, c2);
    const unsigned long long n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += kW0;
    k1 += kW1;
  }
  return Philox4x64Out{{c0, c1, c2, c3}};
}

// Standard Gumbel noise from one 64-bit word: u = (2·(w >> 41) + 1)·2^-24, an
// odd multiple of 2^-24 strictly inside (0, 1) and exact in fp32;
// g = -log(-log u).
__device__ __forceinline__ float gumbel_of_word(unsigned long long w) {
  const float u = (float)(2u * (unsigned)(w >> 41) + 1u) * 0x1p-24f;
  return -logf(-logf(u));
}

template <typename T> struct Num;
template <> struct Num<float> {
  static __device__ __forceinline__ float to_f(float x) { return x; }
  static __device__ __forceinline__ float from_f(float x) { return x; }
  static __device__ __forceinline__ float quant(float x) { return x; }
};
template <> struct Num<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
  static __device__ __forceinline__ float quant(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
  }
};

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide sum for blockDim.x a multiple of 32 (<= 1024).  `red` holds 32 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
  int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float r = (lane < nw) ? red[lane] : 0.f;
  r = warp_sum(r);
  return r;
}
__device__ __forceinline__ float block_max(float v, float* red) {
  int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float r = (lane < nw) ? red[lane] : -INFINITY;
  r = warp_max(r);
  return r;
}

}  // namespace df
