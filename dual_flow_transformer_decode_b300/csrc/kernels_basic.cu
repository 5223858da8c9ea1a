// CUDA-core kernels of the dual-flow decode step: embedding stack, RMSNorm,
// GEMV, the fused GEMM epilogues (QKV + coupling + RoPE + cache append,
// SwiGLU + b coupling, down + c coupling + residual), split-KV attention for
// any head size, the split merge, the softmax/mixture head and the MoE
// router-replay pieces.
//
// Method source: "Resumen Técnico: Dual-Flow Transformers" (gist.science),
// sections "Arquitectura Central" and "Mecanismos Clave".  Stacked rows:
// 0..B-1 primary flow, B..2B-1 auxiliary flow (same sequence order).

#include <algorithm>
#include <math.h>
#include <stdlib.h>

#include <cmath>

#include <cooperative_groups.h>

#include "df_internal.h"
#include "ptx.cuh"

namespace df {

// ------------------------------------------------------------------ position

__global__ void k_set_pos(Ctrl* c, int t) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  c->t = t;
}
// End of a pass: the step counter, the generation history row and, in paged
// mode, the positions of the active sequences in [lo, hi) advance by one.
__global__ void k_advance_pos(Ctrl* c, int* pos, const int* active, int lo, int hi) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  if (threadIdx.x == 0) {
    c->t += 1;
    c->gen_row += 1;
  }
  if (pos)
    for (int b = lo + (int)threadIdx.x; b < hi; b += blockDim.x)
      if (active[b]) pos[b] += 1;
}
__global__ void k_set_seed(Ctrl* c, unsigned long long seed) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  c->seed = seed;
  c->gen_row = 0;
}
// Paged mode: writes up to kIntEdits (index, value) pairs into an int array
// (page-table entries, positions, active flags), in order.
__global__ void k_int_edits(int* dst, IntEdits e) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  if (threadIdx.x == 0)
    for (int i = 0; i < e.n; ++i) dst[e.idx[i]] = e.val[i];
}

template <typename T>
__global__ void k_attn_generic(const T* __restrict__ kv, int layer, KvMap km, const float* __restrict__ qatt,
                               const Ctrl* __restrict__ ctrl, float* __restrict__ part_o,
                               float* __restrict__ part_ml, int B, int Hkv, int G, int hd, int splits, int flo,
                               int fhi);

bool pdl_enabled() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("DF_NO_PDL");
    v = (e && e[0] == '1') ? 0 : 1;
  }
  return v == 1;
}

constexpr int kRouterRows = 4;  // stacked rows per router CTA
template <typename TW, int R>
__global__ void __launch_bounds__(256) k_router(const TW* __restrict__ Wr, const float* __restrict__ un,
                                                float* __restrict__ rlog, int E, int d, int lo, int hi);
template <typename TW>
__global__ void __launch_bounds__(512, 2) k_router_route(
    const TW* __restrict__ Wr, const float* __restrict__ un, int* __restrict__ topk_l, int* __restrict__ topkx,
    float* __restrict__ gate, int* __restrict__ ecount, int* __restrict__ elist, int* __restrict__ eslot,
    int* __restrict__ ticket, int B, int E, int d, int k, int ka, int maxB, int select, int prim, int aux,
    int32_t* __restrict__ dbg_topk_l, float* __restrict__ dbg_router_l);

void kernels_init() {
  cudaFuncSetAttribute(k_attn_generic<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  cudaFuncSetAttribute(k_attn_generic<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  cudaFuncSetAttribute(k_router<__nv_bfloat16, kRouterRows>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       kRouterRows * 8192 * 4);
  cudaFuncSetAttribute(k_router<float, kRouterRows>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       kRouterRows * 8192 * 4);
  cudaFuncSetAttribute(k_router_route<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (2 * 8192 + 2 * 1024) * 4);
  cudaFuncSetAttribute(k_router_route<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (2 * 8192 + 2 * 1024) * 4);
}

void launch_set_pos(Ctrl* c, int t, cudaStream_t s) { launch_pdl(k_set_pos, dim3(1), dim3(1), 0, s, c, t); }
void launch_advance_pos(const Buffers& Bf, int lo, int hi, cudaStream_t s) {
  launch_pdl(k_advance_pos, dim3(1), dim3(128), 0, s, Bf.ctrl, Bf.kvm.table ? Bf.kv_pos : (int*)nullptr,
             (const int*)Bf.kv_active, lo, hi);
}
void launch_int_edits(int* dst, const IntEdits& e, cudaStream_t s) {
  if (e.n > 0) launch_pdl(k_int_edits, dim3(1), dim3(32), 0, s, dst, e);
}
void launch_set_seed(Ctrl* c, unsigned long long seed, cudaStream_t s) {
  launch_pdl(k_set_seed, dim3(1), dim3(1), 0, s, c, seed);
}

// ------------------------------------------------------------------ embedding
// h[b] = E1[x_b], h[B+b] = E2[x_b]: the two flows use separate token
// embeddings of the same token ("Arquitectura Central", Separación).

template <typename T>
__global__ void k_embed(const T* __restrict__ e1, const T* __restrict__ e2, const int32_t* __restrict__ tok,
                        int tok_stride, int use_pos, Ctrl* ctrl, float* __restrict__ h, int B, int lo, int d,
                        int V) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  int m = lo + blockIdx.x;
  int f = m >= B, b = m - f * B;
  int idx = b * tok_stride + (use_pos ? ctrl->t : 0);
  int id = tok[idx];
  bool ok = id >= 0 && id < V;
  if (!ok && threadIdx.x == 0) latch_error(ctrl, kErrDevice, 1000 + b);
  const T* e = (f ? e2 : e1) + (size_t)(ok ? id : 0) * d;
  float* out = h + (size_t)m * d;
  for (int i = threadIdx.x; i < d; i += blockDim.x) out[i] = ok ? Num<T>::to_f(e[i]) : 0.f;
}

void launch_embed(const Dims& D, const Buffers& Bf, const void* emb1, const void* emb2, const int32_t* tokens,
                  int tok_stride, int use_pos, const Rows& R, cudaStream_t s) {
  int n = R.hi - R.lo;
  if (n <= 0) return;
  if (D.bf16)
    launch_pdl(k_embed<__nv_bfloat16>, dim3(n), dim3(256), 0, s, (const __nv_bfloat16*)emb1, (const __nv_bfloat16*)emb2, tokens,
                                              tok_stride, use_pos, Bf.ctrl, Bf.h, R.B, R.lo, D.d, D.V);
  else
    launch_pdl(k_embed<float>, dim3(n), dim3(256), 0, s, (const float*)emb1, (const float*)emb2, tokens, tok_stride, use_pos,
                                     Bf.ctrl, Bf.h, R.B, R.lo, D.d, D.V);
}

// ------------------------------------------------------------------ RMSNorm
// u = x / sqrt(mean(x^2) + eps) * g, rounded to the storage type for the
// next GEMM; optionally also kept unrounded in fp32 (MoE router input).

template <typename T>
__device__ __forceinline__ void store4(T* p, float a, float b, float c, float d);
template <>
__device__ __forceinline__ void store4<float>(float* p, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, float a, float b, float c, float d) {
  __nv_bfloat162* q = reinterpret_cast<__nv_bfloat162*>(p);
  q[0] = __floats2bfloat162_rn(a, b);
  q[1] = __floats2bfloat162_rn(c, d);
}

// One CTA (256 threads) per row; the row is held in registers as float4
// (d <= 8192, d a multiple of 4), so it is read once.
template <typename T>
__global__ void k_rmsnorm(const float* __restrict__ h, const float* __restrict__ g, T* __restrict__ out,
                          float* __restrict__ out_f32, int d, float eps, int lo) {
  __shared__ float red[32];
  const int m = lo + blockIdx.x;
  const float4* x4 = reinterpret_cast<const float4*>(h + (size_t)m * d);
  const float4* g4 = reinterpret_cast<const float4*>(g);
  const int n4 = d >> 2;
  // the gains are fixed inputs: read before the dependency resolves, so only
  // the row load and the reduction sit on the critical path
  float4 gv[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = threadIdx.x + k * 256;
    if (i < n4) gv[k] = g4[i];
  }
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  float4 v[8];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = threadIdx.x + k * 256;
    if (i < n4) {
      v[k] = x4[i];
      ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
    }
  }
  ss = block_sum(ss, red);
  const float r = 1.0f / sqrtf(ss / (float)d + eps);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = threadIdx.x + k * 256;
    if (i < n4) {
      const float4 gg = gv[k];
      const float a = v[k].x * r * gg.x, b = v[k].y * r * gg.y, c = v[k].z * r * gg.z, e = v[k].w * r * gg.w;
      store4<T>(out + (size_t)m * d + 4 * i, a, b, c, e);
      if (out_f32) *reinterpret_cast<float4*>(out_f32 + (size_t)m * d + 4 * i) = make_float4(a, b, c, e);
    }
  }
}

void launch_rmsnorm(const Dims& D, const Buffers& Bf, const float* g, void* out, float* out_f32, const Rows& R,
                    cudaStream_t s) {
  int n = R.hi - R.lo;
  if (n <= 0) return;
  if (D.bf16)
    launch_pdl(k_rmsnorm<__nv_bfloat16>, dim3(n), dim3(256), 0, s, Bf.h, g, (__nv_bfloat16*)out, out_f32, D.d, D.eps, R.lo);
  else
    launch_pdl(k_rmsnorm<float>, dim3(n), dim3(256), 0, s, Bf.h, g, (float*)out, out_f32, D.d, D.eps, R.lo);
}

void launch_rmsnorm_rows(const Dims& D, const float* h, const float* g, void* out, int rows, cudaStream_t s,
                         float* out_f32) {
  if (rows <= 0) return;
  if (D.bf16)
    launch_pdl(k_rmsnorm<__nv_bfloat16>, dim3(rows), dim3(256), 0, s, h, g, (__nv_bfloat16*)out, out_f32, D.d, D.eps,
               0);
  else
    launch_pdl(k_rmsnorm<float>, dim3(rows), dim3(256), 0, s, h, g, (float*)out, out_f32, D.d, D.eps, 0);
}

// ------------------------------------------------------------------ GEMV (CUDA cores)
// The CUDA-core path (fp32 models, and the forced generic sequence): one warp
// per output feature; rows are processed R at a time with one accumulator
// each.  With VEC16, a lane reads 16-byte chunks of the weight row and of
// each activation row (chunk c covers elements 16c/size .. of the row, lane l
// takes chunks l, l + 32, ...), so a warp moves 512 contiguous bytes of the
// weight row per load; otherwise (a row length that is not a whole number of
// chunks) elements are read one by one, lane-strided.  Each row's sum
// depends only on that row, so results do not change with the set of active
// rows.

template <typename T>
__device__ __forceinline__ void unpack16(const uint4& raw, float (&v)[16 / sizeof(T)]);
template <>
__device__ __forceinline__ void unpack16<float>(const uint4& raw, float (&v)[4]) {
  v[0] = __uint_as_float(raw.x);
  v[1] = __uint_as_float(raw.y);
  v[2] = __uint_as_float(raw.z);
  v[3] = __uint_as_float(raw.w);
}
template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4& raw, float (&v)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

template <typename T, int R, bool VEC16>
__global__ void k_gemv(const T* __restrict__ W, int N, int K, const T* __restrict__ X, int ldx,
                       float* __restrict__ out, int ldo, int lo, int hi) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  constexpr int VEC = 16 / sizeof(T);
  int warps = blockDim.x >> 5, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int n = blockIdx.x * warps + w; n < N; n += gridDim.x * warps) {
    const T* wr = W + (size_t)n * K;
    for (int r0 = lo; r0 < hi; r0 += R) {
      float acc[R];
#pragma unroll
      for (int r = 0; r < R; ++r) acc[r] = 0.f;
      if constexpr (VEC16) {
        for (int k0 = lane * VEC; k0 < K; k0 += 32 * VEC) {
          float wv[VEC];
          unpack16<T>(*reinterpret_cast<const uint4*>(wr + k0), wv);
#pragma unroll
          for (int r = 0; r < R; ++r) {
            if (r0 + r < hi) {
              float xv[VEC];
              unpack16<T>(*reinterpret_cast<const uint4*>(X + (size_t)(r0 + r) * ldx + k0), xv);
#pragma unroll
              for (int q = 0; q < VEC; ++q) acc[r] = fmaf(wv[q], xv[q], acc[r]);
            }
          }
        }
      } else {
        for (int k = lane; k < K; k += 32) {
          const float wv = Num<T>::to_f(wr[k]);
#pragma unroll
          for (int r = 0; r < R; ++r)
            if (r0 + r < hi) acc[r] = fmaf(wv, Num<T>::to_f(X[(size_t)(r0 + r) * ldx + k]), acc[r]);
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float v = warp_sum(acc[r]);
        if (lane == 0 && r0 + r < hi) out[(size_t)(r0 + r) * ldo + n] = v;
      }
    }
  }
}

template <typename T>
void launch_gemv_t(const void* W, int N, int K, const void* X, int ldx, float* out, int ldo, const Rows& R,
                   int blocks, cudaStream_t s) {
  constexpr int VEC = 16 / sizeof(T);
  // 16-byte chunks need every weight and activation row to start on a chunk
  // boundary (the buffers themselves are 256-byte aligned)
  if (K % VEC == 0 && ldx % VEC == 0)
    launch_pdl(k_gemv<T, 8, true>, dim3(blocks), dim3(256), 0, s, (const T*)W, N, K, (const T*)X, ldx, out, ldo,
               R.lo, R.hi);
  else
    launch_pdl(k_gemv<T, 8, false>, dim3(blocks), dim3(256), 0, s, (const T*)W, N, K, (const T*)X, ldx, out, ldo,
               R.lo, R.hi);
}

void launch_gemv(const Dims& D, const void* W, int N, int K, const void* X, int ldx, float* out, int ldo,
                 const Rows& R, cudaStream_t s) {
  if (R.hi <= R.lo || N <= 0) return;
  int blocks = (N + 7) / 8;
  if (blocks > 148 * 16) blocks = 148 * 16;
  if (D.bf16)
    launch_gemv_t<__nv_bfloat16>(W, N, K, X, ldx, out, ldo, R, blocks, s);
  else
    launch_gemv_t<float>(W, N, K, X, ldx, out, ldo, R, blocks, s);
}

// ------------------------------------------------------------------ epilogues
// QKV epilogue ("Mecanismos Clave", Atención de KV Compartido Asimétrico):
//  primary row b:   q1 = raw[b][0:qdim] (pre-RoPE), K/V of position t are
//                   RoPE(k1), v1 rounded to the cache type and appended;
//  auxiliary row:   Q2 = raw[B+b][0:qdim] + a ⊙ q1 (coupling before RoPE); its
//                   own K/V columns are discarded (the auxiliary flow writes
//                   no cache);
//  both:            the rotated query is rounded to the cache type.

template <typename T>
__global__ void k_ep_qkv(const float* __restrict__ raw, int ldr, const float* __restrict__ a, T* __restrict__ kv,
                         int layer, KvMap km, const float* __restrict__ rope, const Ctrl* __restrict__ ctrl,
                         float* __restrict__ qatt, Couple C, int B, int lo, int Hq, int Hkv, int hd) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  int m = lo + blockIdx.x;
  int f = m >= B, b = m - f * B;
  int t = kv_seq_pos(km, ctrl, b);
  int half = hd >> 1, qdim = Hq * hd, kvdim = Hkv * hd;
  const float* cs = rope + (size_t)t * hd;
  const float* rr = raw + (size_t)m * ldr;
  for (int p = threadIdx.x; p < Hq * half; p += blockDim.x) {
    int n0 = (p / half) * hd + (p % half), n1 = n0 + half, i = p % half;
    float v0 = rr[n0], v1 = rr[n1];
    if (f) {
      float p0, p1;
      if (C.saved) {
        p0 = C.q1s[(size_t)b * qdim + n0];
        p1 = C.q1s[(size_t)b * qdim + n1];
      } else {
        p0 = raw[(size_t)b * ldr + n0];
        p1 = raw[(size_t)b * ldr + n1];
      }
      v0 = fmaf(a[n0], p0, v0);
      v1 = fmaf(a[n1], p1, v1);
    } else if (C.save) {
      C.q1s[(size_t)b * qdim + n0] = v0;
      C.q1s[(size_t)b * qdim + n1] = v1;
    }
    float c = cs[2 * i], s = cs[2 * i + 1];
    qatt[(size_t)m * qdim + n0] = Num<T>::quant(v0 * c - v1 * s);
    qatt[(size_t)m * qdim + n1] = Num<T>::quant(v1 * c + v0 * s);
  }
  if (f) return;
  const int page = kv_page(km, b, t), off = kv_off(km, t);
  for (int p = threadIdx.x; p < Hkv * half; p += blockDim.x) {
    int g = p / half, i = p % half;
    float k0 = rr[qdim + g * hd + i], k1 = rr[qdim + g * hd + i + half];
    float c = cs[2 * i], s = cs[2 * i + 1];
    T* Kp = kv + kv_index(km, Hkv, hd, layer, 0, page, g, off);
    Kp[i] = Num<T>::from_f(k0 * c - k1 * s);
    Kp[i + half] = Num<T>::from_f(k1 * c + k0 * s);
  }
  for (int p = threadIdx.x; p < kvdim; p += blockDim.x) {
    int g = p / hd, i = p % hd;
    T* Vp = kv + kv_index(km, Hkv, hd, layer, 1, page, g, off);
    Vp[i] = Num<T>::from_f(rr[qdim + kvdim + p]);
  }
}

void launch_ep_qkv(const Dims& D, const Buffers& Bf, const float* raw, int ldr, const float* a, void* kv, int layer,
                   const Couple& C, const Rows& R, cudaStream_t s) {
  int n = R.hi - R.lo;
  if (n <= 0) return;
  if (D.bf16)
    launch_pdl(k_ep_qkv<__nv_bfloat16>, dim3(n), dim3(256), 0, s, raw, ldr, a, (__nv_bfloat16*)kv, layer, Bf.kvm,
               (const float*)Bf.rope, (const Ctrl*)Bf.ctrl, Bf.qatt, C, R.B, R.lo, D.Hq, D.Hkv, D.hd);
  else
    launch_pdl(k_ep_qkv<float>, dim3(n), dim3(256), 0, s, raw, ldr, a, (float*)kv, layer, Bf.kvm,
               (const float*)Bf.rope, (const Ctrl*)Bf.ctrl, Bf.qatt, C, R.B, R.lo, D.Hq, D.Hkv, D.hd);
}

// SwiGLU epilogue with the MLP-intermediate coupling ("Mecanismos Clave",
// Acoplamiento Ligero): z = silu(gate) ⊙ up; auxiliary rows add b ⊙ z1.
// Gate/up rows are interleaved in blocks of 64 (see df_weights.wgu).
template <typename T>
__global__ void k_ep_swiglu(const float* __restrict__ raw, int ldr, const float* __restrict__ bvec,
                            T* __restrict__ z, Couple C, int B, int lo, int F) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  int m = lo + blockIdx.x;
  int f = m >= B, b = m - f * B;
  for (int fi = threadIdx.x; fi < F; fi += blockDim.x) {
    int ng = (fi >> 6) * 128 + (fi & 63), nu = ng + 64;
    float zz = silu_f(raw[(size_t)m * ldr + ng]) * raw[(size_t)m * ldr + nu];
    if (f) {
      float z1 = C.saved ? C.z1s[(size_t)b * F + fi]
                         : silu_f(raw[(size_t)b * ldr + ng]) * raw[(size_t)b * ldr + nu];
      zz = fmaf(bvec[fi], z1, zz);
    } else if (C.save) {
      C.z1s[(size_t)b * F + fi] = zz;
    }
    z[(size_t)m * F + fi] = Num<T>::from_f(zz);
  }
}

void launch_ep_swiglu(const Dims& D, const Buffers& Bf, const float* raw, int ldr, const float* bvec,
                      const Couple& C, const Rows& R, cudaStream_t s) {
  int n = R.hi - R.lo;
  if (n <= 0) return;
  if (D.bf16)
    launch_pdl(k_ep_swiglu<__nv_bfloat16>, dim3(n), dim3(256), 0, s, raw, ldr, bvec, (__nv_bfloat16*)Bf.z, C, R.B, R.lo, D.F);
  else
    launch_pdl(k_ep_swiglu<float>, dim3(n), dim3(256), 0, s, raw, ldr, bvec, (float*)Bf.z, C, R.B, R.lo, D.F);
}

// Down-projection epilogue with the MLP-output coupling: y2 += c ⊙ y1, then
// the residual add h += y for both flows.
__global__ void k_ep_down(const float* __restrict__ raw, int ldr, const float* __restrict__ cvec,
                          float* __restrict__ h, Couple C, int B, int lo, int d) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  int m = lo + blockIdx.x;
  int f = m >= B, b = m - f * B;
  for (int n = threadIdx.x; n < d; n += blockDim.x) {
    float y = raw[(size_t)m * ldr + n];
    if (f) {
      float y1 = C.saved ? C.y1s[(size_t)b * d + n] : raw[(size_t)b * ldr + n];
      y = fmaf(cvec[n], y1, y);
    } else if (C.save) {
      C.y1s[(size_t)b * d + n] = y;
    }
    h[(size_t)m * d + n] += y;
  }
}

void launch_ep_down(const Dims& D, const Buffers& Bf, const float* raw, int ldr, const float* cvec,
                    const Couple& C, const Rows& R, cudaStream_t s) {
  int n = R.hi - R.lo;
  if (n <= 0) return;
  launch_pdl(k_ep_down, dim3(n), dim3(256), 0, s, raw, ldr, cvec, Bf.h, C, R.B, R.lo, D.d);
}

__global__ void k_ep_residual(const float* __restrict__ raw, int ldr, float* __restrict__ h, int lo, int d) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  int m = lo + blockIdx.x;
  for (int n = threadIdx.x; n < d; n += blockDim.x) h[(size_t)m * d + n] += raw[(size_t)m * ldr + n];
}

void launch_ep_residual(const Dims& D, const Buffers& Bf, const float* raw, int ldr, const Rows& R,
                        cudaStream_t s) {
  int n = R.hi - R.lo;
  if (n <= 0) return;
  launch_pdl(k_ep_residual, dim3(n), dim3(256), 0, s, raw, ldr, Bf.h, R.lo, D.d);
}

// ------------------------------------------------------------------ attention
// Split-KV decode attention over the primary cache positions 0..t, shared by
// the primary queries and the auxiliary queries of the same KV head
// ("Mecanismos Clave": the auxiliary flow attends to K1, V1).  Grid: (split,
// kv head, sequence).  Each split keeps a running max m, running sum l and
// unnormalised output o per query row; attn_combine merges the splits.
// Partial slot of a query row: ((b*Hkv + g)*splits + s)*2G + f*G + j.

// Splits per (sequence, KV head), at most 16 (the splits of a pair form one
// thread-block cluster).  Chosen by a simple time model over the cache
// length T (in 64-position tiles): with `slots` = 2 resident CTAs per SM,
//   time(s) = waves(s) * (c0 + ceil(T / s) * c_tile),
//   waves(s) = ceil(pairs * s / slots),
// where c0 (~4 us) is a CTA's fixed cost (barrier set-up, query load, split
// merge) and c_tile (~1.5 us) the time to stream one 32 KB K+V tile at a
// CTA's fair share of HBM bandwidth.
int attn_splits(const Dims& D, int B) {
  const int pairs = B * D.Hkv;
  const int slots = 2 * D.sms;
  const int T = (D.max_len + 63) / 64;
  const double c0 = 4.0, c_tile = 1.5;
  int best = 1;
  double best_t = 1e30;
  for (int s = 1; s <= 16 && s <= T; ++s) {
    const double waves = std::ceil((double)pairs * s / slots);
    const double tm = waves * (c0 + std::ceil((double)T / s) * c_tile);
    if (tm < best_t - 1e-9) {
      best_t = tm;
      best = s;
    }
  }
  return best;
}

__device__ __forceinline__ void split_range(int n, int splits, int s, int& s0, int& s1) {
  int chunk = (n + splits - 1) / splits;
  chunk = (chunk + 63) & ~63;
  s0 = s * chunk;
  s1 = min(n, s0 + chunk);
}

template <typename T>
__global__ void k_attn_generic(const T* __restrict__ kv, int layer, KvMap km, const float* __restrict__ qatt,
                               const Ctrl* __restrict__ ctrl, float* __restrict__ part_o,
                               float* __restrict__ part_ml, int B, int Hkv, int G, int hd, int splits, int flo,
                               int fhi) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  constexpr int CH = 128;  // positions per chunk == blockDim.x
  extern __shared__ float sm[];
  int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  int Ract = (fhi - flo) * G;
  int qdim = Hkv * G * hd;
  float* q = sm;                        // [Ract][hd]
  float* o = q + Ract * hd;             // [Ract][hd]
  float* sc = o + Ract * hd;            // [Ract][CH]
  float* mrow = sc + Ract * CH;         // [Ract]
  float* lrow = mrow + Ract;
  float* corr = lrow + Ract;
  int n = kv_seq_pos(km, ctrl, b) + 1;
  int s0, s1;
  split_range(n, splits, s, s0, s1);
  // key/value row of position p of this (sequence, KV head)
  auto Krow = [&](int p) { return kv + kv_index(km, Hkv, hd, layer, 0, kv_page(km, b, p), g, kv_off(km, p)); };
  auto Vrow = [&](int p) { return kv + kv_index(km, Hkv, hd, layer, 1, kv_page(km, b, p), g, kv_off(km, p)); };
  float scale = 1.0f / sqrtf((float)hd);
  for (int idx = threadIdx.x; idx < Ract * hd; idx += blockDim.x) {
    int r = idx / hd, i = idx % hd;
    int f = flo + r / G, j = r % G;
    q[idx] = qatt[(size_t)(f * B + b) * qdim + (g * G + j) * hd + i];
    o[idx] = 0.f;
  }
  for (int r = threadIdx.x; r < Ract; r += blockDim.x) {
    mrow[r] = -INFINITY;
    lrow[r] = 0.f;
  }
  __syncthreads();
  int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int c0 = s0; c0 < s1; c0 += CH) {
    int pos = c0 + threadIdx.x;
    if (pos < s1) {
      const T* kr = Krow(pos);
      for (int r = 0; r < Ract; ++r) {
        float dot = 0.f;
        for (int i = 0; i < hd; ++i) dot = fmaf(q[r * hd + i], Num<T>::to_f(kr[i]), dot);
        sc[r * CH + threadIdx.x] = dot * scale;
      }
    } else {
      for (int r = 0; r < Ract; ++r) sc[r * CH + threadIdx.x] = -INFINITY;
    }
    __syncthreads();
    for (int r = w; r < Ract; r += nw) {
      float mx = -INFINITY;
      for (int j = lane; j < CH; j += 32) mx = fmaxf(mx, sc[r * CH + j]);
      mx = warp_max(mx);
      float mnew = fmaxf(mrow[r], mx);
      float cf = (mrow[r] == -INFINITY) ? 0.f : expf(mrow[r] - mnew);
      float sum = 0.f;
      for (int j = lane; j < CH; j += 32) {
        float p = (sc[r * CH + j] == -INFINITY) ? 0.f : expf(sc[r * CH + j] - mnew);
        sc[r * CH + j] = p;
        sum += p;
      }
      sum = warp_sum(sum);
      __syncwarp();
      if (lane == 0) {
        lrow[r] = lrow[r] * cf + sum;
        mrow[r] = mnew;
        corr[r] = cf;
      }
    }
    __syncthreads();
    int cnt = min(CH, s1 - c0);
    for (int idx = threadIdx.x; idx < Ract * hd; idx += blockDim.x) {
      int r = idx / hd, i = idx % hd;
      float acc = o[idx] * corr[r];
      for (int j = 0; j < cnt; ++j) acc = fmaf(sc[r * CH + j], Num<T>::to_f(Vrow(c0 + j)[i]), acc);
      o[idx] = acc;
    }
    __syncthreads();
  }
  size_t slot0 = ((size_t)(b * Hkv + g) * splits + s) * (2 * G) + flo * G;
  for (int idx = threadIdx.x; idx < Ract * hd; idx += blockDim.x) part_o[slot0 * hd + idx] = o[idx];
  for (int r = threadIdx.x; r < Ract; r += blockDim.x) {
    part_ml[(slot0 + r) * 2 + 0] = mrow[r];
    part_ml[(slot0 + r) * 2 + 1] = lrow[r];
  }
}

void launch_attention_generic(const Dims& D, const Buffers& Bf, const void* kv, int layer, int splits,
                              const Rows& R, cudaStream_t s) {
  int flo = R.lo >= R.B ? 1 : 0, fhi = R.hi > R.B ? 2 : 1;
  int Ract = (fhi - flo) * D.G;
  size_t smem = (size_t)(Ract * (2 * D.hd + 128) + 3 * Ract) * sizeof(float);
  dim3 grid(splits, D.Hkv, R.B);
  if (D.bf16) {
    launch_pdl(k_attn_generic<__nv_bfloat16>, dim3(grid), dim3(128), smem, s, (const __nv_bfloat16*)kv, layer,
               Bf.kvm, (const float*)Bf.qatt, (const Ctrl*)Bf.ctrl, Bf.part_o, Bf.part_ml, R.B, D.Hkv, D.G, D.hd,
               splits, flo, fhi);
  } else {
    launch_pdl(k_attn_generic<float>, dim3(grid), dim3(128), smem, s, (const float*)kv, layer, Bf.kvm,
               (const float*)Bf.qatt, (const Ctrl*)Bf.ctrl, Bf.part_o, Bf.part_ml, R.B, D.Hkv, D.G, D.hd, splits,
               flo, fhi);
  }
}

// Merge of split partials: o = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s,
// in split order, rounded to the GEMM input type.
template <typename T>
__global__ void k_attn_combine(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                               T* __restrict__ out, int B, int Hkv, int G, int hd, int splits, int flo) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  int b = blockIdx.x, head = blockIdx.y, f = flo + blockIdx.z;
  int g = head / G, j = head % G;
  int qdim = Hkv * G * hd;
  size_t base = (size_t)(b * Hkv + g) * splits * (2 * G) + f * G + j;
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, part_ml[(base + (size_t)s * 2 * G) * 2]);
  float den = 0.f;
  for (int s = 0; s < splits; ++s) {
    float ms = part_ml[(base + (size_t)s * 2 * G) * 2];
    if (ms != -INFINITY) den += expf(ms - M) * part_ml[(base + (size_t)s * 2 * G) * 2 + 1];
  }
  float inv = 1.0f / den;
  for (int i = threadIdx.x; i < hd; i += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < splits; ++s) {
      size_t slot = base + (size_t)s * 2 * G;
      float ms = part_ml[slot * 2];
      if (ms != -INFINITY) acc = fmaf(expf(ms - M), part_o[slot * hd + i], acc);
    }
    out[(size_t)(f * B + b) * qdim + head * hd + i] = Num<T>::from_f(acc * inv);
  }
}

void launch_attn_combine(const Dims& D, const Buffers& Bf, int splits, const Rows& R, cudaStream_t s) {
  int flo = R.lo >= R.B ? 1 : 0, fhi = R.hi > R.B ? 2 : 1;
  dim3 grid(R.B, D.Hq, fhi - flo);
  if (D.bf16)
    launch_pdl(k_attn_combine<__nv_bfloat16>, dim3(grid), dim3(128), 0, s, Bf.part_o, Bf.part_ml, (__nv_bfloat16*)Bf.o, R.B, D.Hkv,
                                                        D.G, D.hd, splits, flo);
  else
    launch_pdl(k_attn_combine<float>, dim3(grid), dim3(128), 0, s, Bf.part_o, Bf.part_ml, (float*)Bf.o, R.B, D.Hkv, D.G, D.hd, splits,
                                               flo);
}

// ------------------------------------------------------------------ mixture head
// p1 = softmax(l1), p2 = softmax(l2), alpha = 0.5 + 0.5 * sum p1^2 (the
// primary's collision probability, so alpha >= 1/2), log p_mix =
// logaddexp(log alpha + log p1, log(1 - alpha) + log p2), argmax with the
// lowest index among equal values ("Mecanismos Clave", Objetivo de Mezcla).

// log(e^x + e^y) with the fast exponential and logarithm: log(1 + e) for
// e = e^(mn - mx) in (0, 1], absolute error a few 1e-7 -- far below the
// bf16-driven deviations of the log-probabilities it produces.
__device__ __forceinline__ float logaddexp_f(float x, float y) {
  if (x == -INFINITY) return y;
  if (y == -INFINITY) return x;
  float mx = fmaxf(x, y), mn = fminf(x, y);
  return mx + __logf(1.0f + __expf(mn - mx));
}

// One cluster of kMixCl CTAs per sequence; CTA r handles the r-th chunk of
// the vocabulary for both flows.  Pass 1 keeps, per thread, online softmax
// statistics relative to a running maximum: flow 1 (max, sum e, sum e^2),
// flow 2 (max, sum e).  The CTAs exchange their block totals through
// distributed shared memory and every CTA merges them in rank order, so all
// of them hold the same row totals.  Pass 2 writes the log-probabilities and
// the per-CTA argmax; rank 0 merges those in rank order.
constexpr int kMixCl = 8;
constexpr int kMixThreads = 256;

struct MixStat {
  float m1, s1, q1, m2, s2;
};

__device__ __forceinline__ void mix_merge(float& m, float& s, float& q, float mo, float so, float qo) {
  if (mo == -INFINITY) return;
  if (m == -INFINITY) {
    m = mo;
    s = so;
    q = qo;
    return;
  }
  const float mn = fmaxf(m, mo);
  const float ea = __expf(m - mn), eb = __expf(mo - mn);
  s = s * ea + so * eb;
  q = q * ea * ea + qo * eb * eb;
  m = mn;
}

__device__ __forceinline__ void mix_merge(MixStat& a, const MixStat& o) {
  mix_merge(a.m1, a.s1, a.q1, o.m1, o.s1, o.q1);
  float dummy = 0.f;
  mix_merge(a.m2, a.s2, dummy, o.m2, o.s2, 0.f);
}

// Online softmax statistics: running max m, sum of e^(x - m) and of
// e^(2(x - m)).  The fast exponential (ex2-based, a few ulp) suffices: the
// sums feed log-probabilities compared at the bf16 level.
__device__ __forceinline__ void mix_push(float& m, float& s, float& q, float x) {
  if (x > m) {
    const float r = __expf(m - x);
    s = s * r + 1.f;
    q = q * r * r + 1.f;
    m = x;
  } else {
    const float e = __expf(x - m);
    s += e;
    q += e * e;
  }
}

__device__ __forceinline__ void argmax_merge(float& best, int& bi, float ov, int oi) {
  if (ov > best || (ov == best && oi < bi)) {
    best = ov;
    bi = oi;
  }
}

// One CTA cluster per sequence b; CTA r of the cluster owns the vocabulary
// chunk [v0, v1).  Pass 1 forms the online (max, Σe, Σe²) statistics of both
// flows' logits, merged over the cluster in rank order.  Pass 2 walks the
// chunk in blocks of 4 tokens (block j holds tokens 4j..4j+3 and belongs to
// the CTA whose chunk holds 4j) and writes log p_mix, tracking its argmax;
// when sampling, the same pass adds one Philox4x64-10 block of Gumbel noise
// per 4 tokens (counter (j, b, t, 0), key (seed, 0)) and tracks the argmax of
// log p_mix + g: one draw from p_mix (Gumbel-max), written to sample_tok[b]
// (the next step's input) and to sample_hist[t][b].
__global__ void __launch_bounds__(kMixThreads) k_mix(const float* __restrict__ logits, int B, int V, int aux_on,
                                                     float* __restrict__ logp_mix, int32_t* __restrict__ argmax,
                                                     float* __restrict__ alpha_out, float* __restrict__ logp1,
                                                     float* __restrict__ logp2, const Ctrl* __restrict__ ctrl,
                                                     KvMap km, int32_t* __restrict__ sample_tok,
                                                     int32_t* __restrict__ sample_hist, int hist_stride) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  __shared__ MixStat wstat[kMixThreads / 32];
  __shared__ MixStat cstat;  // this CTA's block total, read by the whole cluster
  __shared__ float cbest;
  __shared__ int cidx;
  __shared__ float wbest[kMixThreads / 32];
  __shared__ int widx[kMixThreads / 32];
  __shared__ float csbest;
  __shared__ int csidx;
  __shared__ float wsbest[kMixThreads / 32];
  __shared__ int wsidx[kMixThreads / 32];
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int b = blockIdx.y;
  const int r = (int)cl.block_rank();
  const int chunk = (V + kMixCl - 1) / kMixCl;
  const int v0 = r * chunk, v1 = min(V, v0 + chunk);
  const float* l1 = logits + (size_t)b * V;
  const float* l2 = logits + (size_t)(B + b) * V;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;

  MixStat st{-INFINITY, 0.f, 0.f, -INFINITY, 0.f};
  for (int v = v0 + threadIdx.x; v < v1; v += kMixThreads) {
    mix_push(st.m1, st.s1, st.q1, l1[v]);
    if (aux_on) {
      float dummy = 0.f;
      mix_push(st.m2, st.s2, dummy, l2[v]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    MixStat ot{__shfl_xor_sync(0xffffffffu, st.m1, o), __shfl_xor_sync(0xffffffffu, st.s1, o),
               __shfl_xor_sync(0xffffffffu, st.q1, o), __shfl_xor_sync(0xffffffffu, st.m2, o),
               __shfl_xor_sync(0xffffffffu, st.s2, o)};
    mix_merge(st, ot);
  }
  if (lane == 0) wstat[w] = st;
  __syncthreads();
  if (threadIdx.x == 0) {
    MixStat t = wstat[0];
    for (int i = 1; i < kMixThreads / 32; ++i) mix_merge(t, wstat[i]);
    cstat = t;
  }
  cl.sync();
  MixStat tot = *cl.map_shared_rank(&cstat, 0);
  for (int i = 1; i < kMixCl; ++i) mix_merge(tot, *cl.map_shared_rank(&cstat, i));

  const float lse1 = tot.m1 + logf(tot.s1);
  const float lse2 = aux_on ? tot.m2 + logf(tot.s2) : 0.f;
  const float coll = tot.q1 / (tot.s1 * tot.s1);
  const float alpha = aux_on ? 0.5f + 0.5f * coll : 1.0f;
  const float la = logf(alpha);
  const float lb = (alpha < 1.0f) ? log1pf(-alpha) : -INFINITY;
  const bool samp = sample_tok != nullptr;
  const unsigned long long seed = samp ? ctrl->seed : 0ull;
  const int tpos = samp ? kv_seq_pos(km, ctrl, b) : 0;
  const int hrow = samp ? ctrl->gen_row : 0;
  float best = -INFINITY, sbest = -INFINITY;
  int bi = 0x7fffffff, sbi = 0x7fffffff;
  const int jb0 = (v0 + 3) >> 2, jb1 = (v1 + 3) >> 2;
  for (int j = jb0 + threadIdx.x; j < jb1; j += kMixThreads) {
    Philox4x64Out noise{};
    if (samp) noise = philox4x64_10((unsigned long long)j, (unsigned long long)b, (unsigned long long)tpos, 0ull, seed, 0ull);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int v = 4 * j + e;
      if (v >= V) break;
      const float lp1 = l1[v] - lse1;
      float lm = lp1;
      if (aux_on) {
        const float lp2 = l2[v] - lse2;
        lm = logaddexp_f(la + lp1, lb + lp2);
        if (logp2) logp2[(size_t)b * V + v] = lp2;
      }
      if (logp1) logp1[(size_t)b * V + v] = lp1;
      if (logp_mix) logp_mix[(size_t)b * V + v] = lm;
      if (lm > best) {
        best = lm;
        bi = v;
      }
      if (samp) {
        const float key = lm + gumbel_of_word(noise.w[e]);
        if (key > sbest) {
          sbest = key;
          sbi = v;
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    argmax_merge(best, bi, __shfl_xor_sync(0xffffffffu, best, o), __shfl_xor_sync(0xffffffffu, bi, o));
    argmax_merge(sbest, sbi, __shfl_xor_sync(0xffffffffu, sbest, o), __shfl_xor_sync(0xffffffffu, sbi, o));
  }
  if (lane == 0) {
    wbest[w] = best;
    widx[w] = bi;
    wsbest[w] = sbest;
    wsidx[w] = sbi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < kMixThreads / 32; ++i) {
      argmax_merge(best, bi, wbest[i], widx[i]);
      argmax_merge(sbest, sbi, wsbest[i], wsidx[i]);
    }
    cbest = best;
    cidx = bi;
    csbest = sbest;
    csidx = sbi;
  }
  cl.sync();
  if (r == 0 && threadIdx.x == 0) {
    float cb = cbest, sb = csbest;
    int ci = cidx, si = csidx;
    for (int i = 1; i < kMixCl; ++i) {
      argmax_merge(cb, ci, *cl.map_shared_rank(&cbest, i), *cl.map_shared_rank(&cidx, i));
      argmax_merge(sb, si, *cl.map_shared_rank(&csbest, i), *cl.map_shared_rank(&csidx, i));
    }
    if (argmax) argmax[b] = ci;
    if (alpha_out) alpha_out[b] = alpha;
    if (samp) {
      sample_tok[b] = si;
      if (sample_hist) sample_hist[(size_t)hrow * hist_stride + b] = si;
    }
  }
  // keep every CTA's shared memory alive until rank 0 has read it
  cl.sync();
}

void launch_mix(const Dims& D, const Buffers& Bf, int B, int aux_on, float* logp_mix, int32_t* argmax, float* alpha,
                float* logp1, float* logp2, int32_t* sample_tok, int32_t* sample_hist, cudaStream_t s) {
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(kMixCl, B);
  lc.blockDim = dim3(kMixThreads);
  lc.dynamicSmemBytes = 0;
  lc.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kMixCl;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  lc.attrs = at;
  lc.numAttrs = 2;
  cudaLaunchKernelEx(&lc, k_mix, (const float*)Bf.logits, B, D.V, aux_on, logp_mix, argmax, alpha, logp1, logp2,
                     (const Ctrl*)Bf.ctrl, Bf.kvm, sample_tok, sample_hist, D.maxB);
}

// ------------------------------------------------------------------ MoE (router replay)
// Router logits r[m][e] = Wr[e] · un[m] with the normed row unrounded (fp32)
// and Wr stored in the weight type.  CTA (row block, expert block): up to
// kRouterRows consecutive stacked rows held in shared memory, warp w computes
// expert 8*blockIdx.y + w for all of them with 16-byte weight loads (each
// weight vector is read once per row block).
template <typename TW, int R>
__global__ void __launch_bounds__(256) k_router(const TW* __restrict__ Wr, const float* __restrict__ un,
                                                float* __restrict__ rlog, int E, int d, int lo, int hi) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  extern __shared__ float xrows[];  // [R][d]
  const int m0 = lo + blockIdx.x * R;
  const int nr = min(R, hi - m0);
  {
    // 16-byte copies, a batch of loads in flight before the stores (d is a
    // multiple of 8)
    const float4* src = reinterpret_cast<const float4*>(un + (size_t)m0 * d);
    float4* dst = reinterpret_cast<float4*>(xrows);
    const int n4 = nr * d / 4;
    for (int i0 = threadIdx.x; i0 < n4; i0 += 8 * blockDim.x) {
      float4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = i0 + j * blockDim.x;
        if (i < n4) v[j] = src[i];
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = i0 + j * blockDim.x;
        if (i < n4) dst[i] = v[j];
      }
    }
  }
  __syncthreads();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.y * 8 + w;
  if (e >= E) return;
  constexpr int VEC = 16 / sizeof(TW);
  const TW* wr = Wr + (size_t)e * d;
  float acc[R];
#pragma unroll
  for (int r = 0; r < R; ++r) acc[r] = 0.f;
  for (int k0 = lane * VEC; k0 < d; k0 += 32 * VEC) {
    const uint4 raw = *reinterpret_cast<const uint4*>(wr + k0);
    const TW* wv = reinterpret_cast<const TW*>(&raw);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (r >= nr) break;
      // the row's VEC values as float4s (same summation order as scalar reads)
      float xv[VEC];
#pragma unroll
      for (int q4 = 0; q4 < VEC / 4; ++q4) {
        const float4 x = *reinterpret_cast<const float4*>(xrows + r * d + k0 + 4 * q4);
        xv[4 * q4] = x.x;
        xv[4 * q4 + 1] = x.y;
        xv[4 * q4 + 2] = x.z;
        xv[4 * q4 + 3] = x.w;
      }
#pragma unroll
      for (int q = 0; q < VEC; ++q) acc[r] = fmaf(Num<TW>::to_f(wv[q]), xv[q], acc[r]);
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (r >= nr) break;
    const float v = warp_sum(acc[r]);
    if (lane == 0) rlog[(size_t)(m0 + r) * E + e] = v;
  }
}

void launch_router_rows(const Dims& D, const void* Wr, const float* un, float* rlog, int rows, cudaStream_t s) {
  if (rows <= 0) return;
  const dim3 grid((rows + kRouterRows - 1) / kRouterRows, (D.E + 7) / 8);
  const size_t smem = (size_t)kRouterRows * D.d * sizeof(float);
  if (D.bf16)
    launch_pdl(k_router<__nv_bfloat16, kRouterRows>, grid, dim3(256), smem, s, (const __nv_bfloat16*)Wr, un, rlog,
               D.E, D.d, 0, rows);
  else
    launch_pdl(k_router<float, kRouterRows>, grid, dim3(256), smem, s, (const float*)Wr, un, rlog, D.E, D.d, 0, rows);
}

// The primary rows choose their top-k experts (descending router logit,
// ties to the lower index); each flow's gates are the softmax of its own
// router logits over that set ("Mecanismos Clave", Replay de Router).  With
// an independent auxiliary fan-out (ka > k; "Contribuciones Clave" 3) the
// auxiliary row also takes its own ka - k largest router logits among the
// other experts, and its gates are the softmax over the replayed set
// followed by those.  Entries: b*k + j (replayed; both flows' rows) and
// B*k + b*(ka-k) + j (auxiliary-own; the auxiliary row only).  The
// per-expert entry lists (ascending entry) let every selected expert's
// weights be read once for all rows that use it; an expert is either
// replayed or auxiliary-own for a sequence, never both, so a list holds at
// most B entries.

// Warp-wide argmax over experts e = lane, lane+32, ... not in the taken
// bitmasks (larger value wins, equal values -> lower index).
__device__ __forceinline__ int warp_pick(const float* r, int E, int lane, unsigned long long tlo,
                                         unsigned long long thi) {
  float best = -INFINITY;
  int bi = 0x7fffffff;
  int q = 0;
  for (int e = lane; e < E; e += 32, ++q) {
    const bool tk = q < 64 ? ((tlo >> q) & 1ull) : ((thi >> (q - 64)) & 1ull);
    if (tk) continue;
    const float v = r[e];
    if (v > best || (v == best && e < bi)) {
      best = v;
      bi = e;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > best || (ov == best && oi < bi)) {
      best = ov;
      bi = oi;
    }
  }
  return bi;
}

__device__ __forceinline__ void mark_taken(int e, int lane, unsigned long long& tlo, unsigned long long& thi) {
  if (e != 0x7fffffff && (e % 32) == lane) {
    const int qq = e / 32;
    if (qq < 64)
      tlo |= 1ull << qq;
    else
      thi |= 1ull << (qq - 64);
  }
}

// Softmax gates of `n` entries held by lanes 0..n-1 (max and sum in entry order).
__device__ __forceinline__ float entry_gate(float v, int n, int lane) {
  float mx = -INFINITY;
  for (int j = 0; j < n; ++j) mx = fmaxf(mx, __shfl_sync(0xffffffffu, v, j));
  const float ex = lane < n ? expf(v - mx) : 0.f;
  float den = 0.f;
  for (int j = 0; j < n; ++j) den += __shfl_sync(0xffffffffu, ex, j);
  return ex / den;
}


// Router logits and routing in one launch.  A cluster of kRouteCl CTAs
// serves sequence b: CTA r computes the router logits of the sequence's
// active rows (primary b, auxiliary B + b) for its share of the experts,
// with the same per-(row, expert) arithmetic as k_router; rank 0 gathers the
// logits through distributed shared memory and routes the sequence as
// described above.  The last rank-0 CTA to finish (a ticket counter in
// global memory, reset by that CTA) builds the per-expert entry lists from
// every sequence's selection.
constexpr int kRouteThreads = 512;
constexpr int kRouteCl = 4;     // CTAs per sequence (cluster)
constexpr int kRouteBatch = 8;  // 16-byte weight loads of one lane in flight at once

template <typename TW>
__global__ void __launch_bounds__(kRouteThreads, 2) k_router_route(
    const TW* __restrict__ Wr, const float* __restrict__ un, int* __restrict__ topk_l, int* __restrict__ topkx,
    float* __restrict__ gate, int* __restrict__ ecount, int* __restrict__ elist, int* __restrict__ eslot,
    int* __restrict__ ticket, int B, int E, int d, int k, int ka, int maxB, int select, int prim, int aux,
    int32_t* __restrict__ dbg_topk_l, float* __restrict__ dbg_router_l) {
  // [2][d] the sequence's rows (primary, auxiliary), then (last CTA) the
  // entries; [2][E] router logits (this CTA's experts; rank 0: all)
  extern __shared__ float rsm_raw[];
  float* xr = rsm_raw;
  float* rsm = rsm_raw + 2 * d;
  __shared__ int last;
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int rank = (int)cl.block_rank(), b = blockIdx.y;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, warps = kRouteThreads / 32;
  const int kx = aux ? ka - k : 0;  // auxiliary-own experts per token
  const int per = (E + kRouteCl - 1) / kRouteCl, e0 = rank * per, e1 = min(E, e0 + per);
  {
    const int n4 = d / 4;
    const float4* s0 = reinterpret_cast<const float4*>(un + (size_t)b * d);
    const float4* s1 = reinterpret_cast<const float4*>(un + (size_t)(B + b) * d);
    float4* d4 = reinterpret_cast<float4*>(xr);
    for (int i = threadIdx.x; i < n4; i += kRouteThreads) {
      if (prim) d4[i] = s0[i];
      if (aux) d4[n4 + i] = s1[i];
    }
  }
  __syncthreads();
  // ---- logits of experts e0 + w, e0 + w + 16, ... for both rows, with
  // kRouteBatch weight loads per lane in flight
  constexpr int VEC = 16 / sizeof(TW);
  for (int e = e0 + w; e < e1; e += warps) {
    const TW* wr = Wr + (size_t)e * d;
    float acc0 = 0.f, acc1 = 0.f;
    for (int c0 = 0; c0 < d; c0 += 32 * VEC * kRouteBatch) {
      uint4 raw[kRouteBatch];
#pragma unroll
      for (int t = 0; t < kRouteBatch; ++t) {
        const int k0 = c0 + (t * 32 + lane) * VEC;
        if (k0 < d) raw[t] = *reinterpret_cast<const uint4*>(wr + k0);
      }
#pragma unroll
      for (int t = 0; t < kRouteBatch; ++t) {
        const int k0 = c0 + (t * 32 + lane) * VEC;
        if (k0 >= d) break;
        const TW* wv = reinterpret_cast<const TW*>(&raw[t]);
        if (prim) {
#pragma unroll
          for (int q4 = 0; q4 < VEC / 4; ++q4) {
            const float4 x = *reinterpret_cast<const float4*>(xr + k0 + 4 * q4);
            acc0 = fmaf(Num<TW>::to_f(wv[4 * q4]), x.x, acc0);
            acc0 = fmaf(Num<TW>::to_f(wv[4 * q4 + 1]), x.y, acc0);
            acc0 = fmaf(Num<TW>::to_f(wv[4 * q4 + 2]), x.z, acc0);
            acc0 = fmaf(Num<TW>::to_f(wv[4 * q4 + 3]), x.w, acc0);
          }
        }
        if (aux) {
#pragma unroll
          for (int q4 = 0; q4 < VEC / 4; ++q4) {
            const float4 x = *reinterpret_cast<const float4*>(xr + d + k0 + 4 * q4);
            acc1 = fmaf(Num<TW>::to_f(wv[4 * q4]), x.x, acc1);
            acc1 = fmaf(Num<TW>::to_f(wv[4 * q4 + 1]), x.y, acc1);
            acc1 = fmaf(Num<TW>::to_f(wv[4 * q4 + 2]), x.z, acc1);
            acc1 = fmaf(Num<TW>::to_f(wv[4 * q4 + 3]), x.w, acc1);
          }
        }
      }
    }
    acc0 = warp_sum(acc0);
    acc1 = warp_sum(acc1);
    if (lane == 0) {
      rsm[e] = acc0;
      rsm[E + e] = acc1;
    }
  }
  cl.sync();
  if (rank == 0) {
    for (int i = threadIdx.x; i < 2 * E; i += kRouteThreads) {
      const int e = i < E ? i : i - E, owner = e / per;
      if (owner != 0) rsm[i] = cl.map_shared_rank(rsm, owner)[i];
    }
  }
  // the other ranks' logits stay readable until rank 0 has copied them
  cl.sync();
  if (rank != 0) return;
  // ---- routing of sequence b (warp 0 of rank 0)
  if (w == 0) {
    int sel = 0;  // lane j < k: the j-th replayed expert
    unsigned long long tlo = 0ull, thi = 0ull;
    if (select) {
      for (int j = 0; j < k; ++j) {
        const int bi = warp_pick(rsm, E, lane, tlo, thi);
        if (lane == 0) topk_l[b * k + j] = bi;
        if (lane == j) sel = bi;
        mark_taken(bi, lane, tlo, thi);
      }
    } else {
      if (lane < k) sel = topk_l[b * k + lane];
      for (int j = 0; j < k; ++j) mark_taken(__shfl_sync(0xffffffffu, sel, j), lane, tlo, thi);
    }
    if (prim) {
      const float g = entry_gate(lane < k ? rsm[sel] : -INFINITY, k, lane);
      if (lane < k) gate[(size_t)b * ka + lane] = g;
    }
    int own = 0;  // lane k + j: the j-th auxiliary-own expert
    if (aux) {
      const float* r = rsm + E;
      for (int j = 0; j < kx; ++j) {
        const int bi = warp_pick(r, E, lane, tlo, thi);
        if (lane == 0) topkx[b * kx + j] = bi;
        if (lane == k + j) own = bi;
        mark_taken(bi, lane, tlo, thi);
      }
      const int ent = lane < k ? sel : own;
      const float g = entry_gate(lane < k + kx ? r[ent] : -INFINITY, k + kx, lane);
      if (lane < k + kx) gate[(size_t)(B + b) * ka + lane] = g;
      if (dbg_topk_l && lane >= k && lane < k + kx) dbg_topk_l[b * ka + lane] = own;
    }
    if (dbg_topk_l && prim && lane < k) dbg_topk_l[b * ka + lane] = sel;
    if (dbg_router_l && prim)
      for (int e = lane; e < E; e += 32) dbg_router_l[(size_t)b * E + e] = rsm[e];
    // this sequence's selection is visible device-wide before the ticket
    __threadfence();
    __syncwarp();
    if (lane == 0) last = atomicAdd(ticket, 1) == (int)gridDim.y - 1;  // one arrival per sequence
  }
  __syncthreads();
  if (!last) return;
  // ---- the last CTA: entry lists in ascending entry order, warp per expert
  __threadfence();
  if (threadIdx.x == 0) *ticket = 0;
  const int nent = B * k + B * kx;
  const bool staged = nent <= 2 * d;
  int* ents = reinterpret_cast<int*>(xr);
  if (staged) {
    for (int i = threadIdx.x; i < nent; i += kRouteThreads)
      ents[i] = i < B * k ? __ldcg(topk_l + i) : __ldcg(topkx + i - B * k);
    __syncthreads();
  }
  for (int e = w; e < E; e += warps) {
    int cnt = 0;
    for (int base = 0; base < nent; base += 32) {
      const int idx = base + lane;
      const int ex = idx >= nent ? -1 : staged ? ents[idx] : idx < B * k ? __ldcg(topk_l + idx) : __ldcg(topkx + idx - B * k);
      const bool hit = idx < nent && ex == e;
      const unsigned m = __ballot_sync(0xffffffffu, hit);
      if (hit) {
        const int slot = cnt + __popc(m & ((1u << lane) - 1u));
        eslot[idx] = slot;
        elist[(size_t)e * maxB + slot] = idx;
      }
      cnt += __popc(m);
    }
    if (lane == 0) ecount[e] = cnt;
  }
}

void launch_router_route(const Dims& D, const Buffers& Bf, const void* Wr, int layer, int select, const Rows& R,
                         int32_t* dbg_topk, float* dbg_router, cudaStream_t s) {
  int* topk_l = Bf.topk + (size_t)layer * D.maxB * D.k;
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(kRouteCl, R.B);
  lc.blockDim = dim3(kRouteThreads);
  lc.dynamicSmemBytes = (size_t)(2 * D.d + 2 * D.E) * sizeof(float);  // d <= 8192, E <= 1024: at most 72 KB
  lc.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kRouteCl;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  lc.attrs = at;
  lc.numAttrs = 2;
  int32_t* dt = dbg_topk ? dbg_topk + (size_t)layer * R.B * D.ka : nullptr;
  float* dr = dbg_router ? dbg_router + (size_t)layer * R.B * D.E : nullptr;
  const int prim = R.has_primary() ? 1 : 0, aux = R.has_aux() ? 1 : 0;
  if (D.bf16)
    cudaLaunchKernelEx(&lc, k_router_route<__nv_bfloat16>, (const __nv_bfloat16*)Wr, (const float*)Bf.un, topk_l,
                       Bf.topkx, Bf.gate, Bf.ecount, Bf.elist, Bf.eslot, Bf.ticket, R.B, D.E, D.d, D.k, D.ka, D.maxB,
                       select, prim, aux, dt, dr);
  else
    cudaLaunchKernelEx(&lc, k_router_route<float>, (const float*)Wr, (const float*)Bf.un, topk_l, Bf.topkx, Bf.gate,
                       Bf.ecount, Bf.elist, Bf.eslot, Bf.ticket, R.B, D.E, D.d, D.k, D.ka, D.maxB, select, prim, aux,
                       dt, dr);
}

// Expert gate/up + SwiGLU + b coupling (CUDA cores): one warp per expert
// hidden unit, looping over the expert's entries and the active flows.
template <typename T>
__global__ void k_moe_gateup(const T* __restrict__ wgu, const float* __restrict__ bvec, const T* __restrict__ u,
                             const int* __restrict__ ecount, const int* __restrict__ elist, T* __restrict__ zE,
                             Couple C, int B, int d, int Fe, int k, int ka, int maxB, int prim, int aux) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  int e = blockIdx.x;
  int cnt = ecount[e];
  if (cnt == 0) return;
  int warps = blockDim.x >> 5, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int fi = blockIdx.y * warps + w;
  if (fi >= Fe) return;
  const T* W = wgu + (size_t)e * 2 * Fe * d;
  const T* wg = W + (size_t)((fi >> 6) * 128 + (fi & 63)) * d;
  const T* wu = wg + (size_t)64 * d;
  for (int idx = 0; idx < cnt; ++idx) {
    const int ent = elist[(size_t)e * maxB + idx];
    // replayed entry (both flows) or auxiliary-own entry (auxiliary row only)
    const bool own = ent >= B * k;
    const int b = own ? (ent - B * k) / (ka - k) : ent / k;
    const int j = own ? k + (ent - B * k) % (ka - k) : ent % k;
    float z1 = 0.f;
    for (int f = (prim && !own) ? 0 : 1; f < (aux ? 2 : 1); ++f) {
      const T* x = u + (size_t)(f * B + b) * d;
      float ag = 0.f, au = 0.f;
      for (int kk = lane; kk < d; kk += 32) {
        float xv = Num<T>::to_f(x[kk]);
        ag = fmaf(Num<T>::to_f(wg[kk]), xv, ag);
        au = fmaf(Num<T>::to_f(wu[kk]), xv, au);
      }
      ag = warp_sum(ag);
      au = warp_sum(au);
      float zz = silu_f(ag) * au;
      if (f == 0) {
        z1 = zz;
        if (C.save && lane == 0) C.z1s[(size_t)ent * Fe + fi] = zz;
      } else if (!own) {  // the b coupling exists for replayed experts only
        float p = C.saved ? C.z1s[(size_t)ent * Fe + fi] : z1;
        zz = fmaf(bvec[fi], p, zz);
      }
      if (lane == 0) zE[((size_t)(f * maxB + b) * ka + j) * Fe + fi] = Num<T>::from_f(zz);
    }
  }
}

void launch_moe_gateup_generic(const Dims& D, const Buffers& Bf, const void* wgu, const float* bvec,
                               const Couple& C, const Rows& R, cudaStream_t s) {
  dim3 grid(D.E, (D.Fe + 7) / 8);
  if (D.bf16)
    launch_pdl(k_moe_gateup<__nv_bfloat16>, dim3(grid), dim3(256), 0, s, (const __nv_bfloat16*)wgu, bvec, (const __nv_bfloat16*)Bf.u,
                                                      Bf.ecount, Bf.elist, (__nv_bfloat16*)Bf.zE, C, R.B, D.d,
                                                      D.Fe, D.k, D.ka, D.maxB, R.has_primary(), R.has_aux());
  else
    launch_pdl(k_moe_gateup<float>, dim3(grid), dim3(256), 0, s, (const float*)wgu, bvec, (const float*)Bf.u, Bf.ecount, Bf.elist,
                                             (float*)Bf.zE, C, R.B, D.d, D.Fe, D.k, D.ka, D.maxB, R.has_primary(),
                                             R.has_aux());
}

template <typename T>
__global__ void k_moe_down(const T* __restrict__ wd, const T* __restrict__ zE, const int* __restrict__ ecount,
                           const int* __restrict__ elist, float* __restrict__ yE, int B, int d, int Fe, int k, int ka,
                           int maxB, int prim, int aux) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  int e = blockIdx.x;
  int cnt = ecount[e];
  if (cnt == 0) return;
  int warps = blockDim.x >> 5, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int n = blockIdx.y * warps + w;
  if (n >= d) return;
  const T* wr = wd + ((size_t)e * d + n) * Fe;
  for (int idx = 0; idx < cnt; ++idx) {
    const int ent = elist[(size_t)e * maxB + idx];
    const bool own = ent >= B * k;
    const int b = own ? (ent - B * k) / (ka - k) : ent / k;
    const int j = own ? k + (ent - B * k) % (ka - k) : ent % k;
    for (int f = (prim && !own) ? 0 : 1; f < (aux ? 2 : 1); ++f) {
      const T* z = zE + ((size_t)(f * maxB + b) * ka + j) * Fe;
      float acc = 0.f;
      for (int kk = lane; kk < Fe; kk += 32) acc = fmaf(Num<T>::to_f(wr[kk]), Num<T>::to_f(z[kk]), acc);
      acc = warp_sum(acc);
      if (lane == 0) yE[((size_t)(f * maxB + b) * ka + j) * d + n] = acc;
    }
  }
}

void launch_moe_down_generic(const Dims& D, const Buffers& Bf, const void* wd, const Rows& R, cudaStream_t s) {
  dim3 grid(D.E, (D.d + 7) / 8);
  if (D.bf16)
    launch_pdl(k_moe_down<__nv_bfloat16>, dim3(grid), dim3(256), 0, s, (const __nv_bfloat16*)wd, (const __nv_bfloat16*)Bf.zE,
                                                    Bf.ecount, Bf.elist, Bf.yE, R.B, D.d, D.Fe, D.k, D.ka,
                                                    D.maxB, R.has_primary(), R.has_aux());
  else
    launch_pdl(k_moe_down<float>, dim3(grid), dim3(256), 0, s, (const float*)wd, (const float*)Bf.zE, Bf.ecount, Bf.elist, Bf.yE, R.B,
                                           D.d, D.Fe, D.k, D.ka, D.maxB, R.has_primary(), R.has_aux());
}

// y_f = sum_j gate_f[j] * yE_f[j] (slot order), y2 += c ⊙ y1, h += y.
__global__ void k_moe_combine(const float* __restrict__ yE, const float* __restrict__ gate,
                              const float* __restrict__ cvec, float* __restrict__ h, Couple C, int B, int lo, int d,
                              int k, int ka, int maxB) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  int m = lo + blockIdx.x;
  int f = m >= B, b = m - f * B;
  const int kr = f ? ka : k;  // entries of this row: the replayed ones, then the auxiliary-own ones
  for (int n = threadIdx.x; n < d; n += blockDim.x) {
    float y = 0.f;
    for (int j = 0; j < kr; ++j)
      y = fmaf(gate[(size_t)m * ka + j], yE[((size_t)(f * maxB + b) * ka + j) * d + n], y);
    if (f) {
      float y1;
      if (C.saved) {
        y1 = C.y1s[(size_t)b * d + n];
      } else {
        y1 = 0.f;
        for (int j = 0; j < k; ++j) y1 = fmaf(gate[(size_t)b * ka + j], yE[((size_t)b * ka + j) * d + n], y1);
      }
      y = fmaf(cvec[n], y1, y);
    } else if (C.save) {
      C.y1s[(size_t)b * d + n] = y;
    }
    h[(size_t)m * d + n] += y;
  }
}

void launch_moe_combine(const Dims& D, const Buffers& Bf, const float* cvec, const Couple& C, const Rows& R,
                        cudaStream_t s) {
  int n = R.hi - R.lo;
  if (n <= 0) return;
  launch_pdl(k_moe_combine, dim3(n), dim3(256), 0, s, Bf.yE, Bf.gate, cvec, Bf.h, C, R.B, R.lo, D.d, D.k, D.ka,
             D.maxB);
}

}  // namespace df
