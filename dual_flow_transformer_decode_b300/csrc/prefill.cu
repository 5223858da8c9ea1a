// Batched (chunked) prefill of the primary flow for dense bf16 models with
// head_dim 128.
//
// "Arquitectura Central" ("Resumen Técnico: Dual-Flow Transformers"): prefill
// runs the primary flow alone, as a standard causal Transformer, and writes
// the one persistent KV cache; the auxiliary flow starts at the first decode
// step.  Instead of one full pass per prompt position, the prompt is taken a
// chunk of positions at a time, B x C rows per chunk (C = rows / B), and every
// layer runs once per chunk:
//
//   embed -> per layer [RMSNorm, QKV GEMM (+ RoPE, bf16 queries, K/V appended
//   at each row's position), causal attention over the cache, Wo GEMM +
//   residual, RMSNorm, gate/up GEMM (+ SwiGLU), down GEMM + residual]
//
// GEMMs: D[128 rows][128 features] = X_tile · W_tile^T on tcgen05 (kind::f16,
// fp32 accumulator of 128 TMEM columns), both operands staged by TMA in the
// 128-byte-swizzled layout through a 6-stage mbarrier ring, one CTA per
// (row tile, feature tile) with the row tile varying fastest so the CTAs that
// share a weight tile run together and hit L2.  Each epilogue thread owns one
// activation row and all 128 features of the tile, so RoPE pairs (j, j+64)
// and gate/up pairs are local.
//
// Attention: one CTA per (64-query block, query head, sequence); a producer
// warp streams 64-position K and V tiles of the sequence's KV head from the
// cache (positions of earlier chunks included) by TMA, four warps each own 16
// queries and run S = Q·K^T and O += P·V on mma.sync m16n8k16 with an online
// softmax and the causal mask; P enters as bf16 hi + lo parts, as in the
// decode kernel.
//
// Quantisation points are those of the decode step: GEMM inputs, cache
// stores and queries in bf16, residual and softmax in fp32.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>

#include "attn_fast.h"
#include "prefill.h"
#include "ptx.cuh"
#include "tc_gemm.h"
#include "tc_moe.h"

namespace df {

namespace {

constexpr int kBM = 128;                 // activation rows per tile
constexpr int kBN = 128;                 // output features per tile
constexpr int kBK = 64;
constexpr int kStageA = kBM * kBK * 2;   // 16 KB
constexpr int kStageB = kBN * kBK * 2;   // 16 KB
constexpr int kStage = kStageA + kStageB;
constexpr int kStages = 6;
constexpr int kChunkRows = 2048;
constexpr int kHD = 128;

enum : int { BP_QKV = 0, BP_RESID = 1, BP_SWIGLU = 2, BP_YOUT = 3 };

struct BpEp {
  int op;
  int Mc, C, p0;        // rows of the chunk, positions per sequence in it, first position
  __nv_bfloat16* q;     // [rows][qdim] rotated queries
  int qdim, kvdim;
  __nv_bfloat16* kv;    // the cache (all layers)
  int layer;
  KvMap km;             // cache addressing
  int slot0;            // cache sequence of the chunk's sequence 0
  int Hkv;
  const float* rope;    // [max_len][hd/2][2]
  float* h;             // residual rows [rows][d]
  int d;
  __nv_bfloat16* z;     // SwiGLU output [rows][F]
  int F;
  // Grouped expert GEMMs (MoE): row tile rt of the launch is entry rt of the
  // block table gblk[rt] = (expert, first packed row), expert -1 meaning no
  // block; the weights of expert e start at weight row e * wrows.
  const int* gblk;
  int wrows;
  float* y;             // BP_YOUT: fp32 output rows [rows][ldy]
  int ldy;
};

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 16 consecutive bf16 values (two 16-byte stores).
__device__ __forceinline__ void store16(__nv_bfloat16* dst, const float (&v)[16]) {
  uint4 a, b;
  a.x = pack2(v[0], v[1]);
  a.y = pack2(v[2], v[3]);
  a.z = pack2(v[4], v[5]);
  a.w = pack2(v[6], v[7]);
  b.x = pack2(v[8], v[9]);
  b.y = pack2(v[10], v[11]);
  b.z = pack2(v[12], v[13]);
  b.w = pack2(v[14], v[15]);
  reinterpret_cast<uint4*>(dst)[0] = a;
  reinterpret_cast<uint4*>(dst)[1] = b;
}

__device__ __forceinline__ void add16(float* dst, const float (&v)[16]) {
  float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float4 x = d4[k];
    x.x += v[4 * k];
    x.y += v[4 * k + 1];
    x.z += v[4 * k + 2];
    x.w += v[4 * k + 3];
    d4[k] = x;
  }
}

__global__ void __launch_bounds__(128, 1)
    k_bp_gemm(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap tw, int kblocks, BpEp ep,
              Ctrl* ctrl) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(base + (size_t)kStages * kStage);
  uint64_t* empty = full + kStages;
  uint64_t* done = empty + kStages;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* flags = reinterpret_cast<volatile int*>(tslot + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rt = blockIdx.x, ft = blockIdx.y;
  // activation rows and weight rows of this tile
  int xrow0 = rt * kBM, wrow0 = ft * kBN;
  if (ep.gblk) {
    // the block table comes from the previous kernel; a tile past the table's
    // end leaves before taking any resource
    ptx::grid_dep_wait();
    const int ex = ep.gblk[2 * rt];
    if (ex < 0) return;  // uniform across the CTA
    xrow0 = ep.gblk[2 * rt + 1];
    wrow0 = ex * ep.wrows + ft * kBN;
  }
  if (tid == 0) {
    ptx::prefetch_tmap(&tx);
    ptx::prefetch_tmap(&tw);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(done, 1);
    flags[0] = 0;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 0) {
    ptx::tmem_alloc(tslot, kBN);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tslot;
  ptx::grid_dep_wait();

  if (warp == 0 && lane == 0) {
    int issued = 0;
    for (int i = 0; i < kblocks; ++i) {
      const int s = i % kStages;
      if (i >= kStages && !ptx::mbar_wait(&empty[s], ((i / kStages) - 1) & 1)) {
        flags[0] = 1;
        latch_error(ctrl, kErrTimeout, 400);
        break;
      }
      uint8_t* a = base + (size_t)s * kStage;
      ptx::mbar_arrive_expect_tx(&full[s], kStage);
      ptx::tma_load_2d(a, &tx, &full[s], i * kBK, xrow0);
      ptx::tma_load_2d(a + kStageA, &tw, &full[s], i * kBK, wrow0);
      issued = i + 1;
    }
    if (flags[0]) {
      // let copies still in flight land before the shared memory is released
      for (int i = issued - kStages < 0 ? 0 : issued - kStages; i < issued; ++i)
        ptx::mbar_wait(&full[i % kStages], (i / kStages) & 1, 100000000ull);
    }
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = ptx::idesc_bf16_f32(kBM, kBN);
    for (int i = 0; i < kblocks; ++i) {
      const int s = i % kStages;
      if (!ptx::mbar_wait(&full[s], (i / kStages) & 1)) {
        flags[0] = 1;
        latch_error(ctrl, kErrTimeout, 401);
        break;
      }
      if (flags[0]) break;
      ptx::tc_fence_after();
      const uint32_t a0 = ptx::smem_u32(base + (size_t)s * kStage), b0 = a0 + kStageA;
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk)
        ptx::mma_bf16(tmem, ptx::desc_sw128(a0 + kk * 32), ptx::desc_sw128(b0 + kk * 32), idesc,
                      (i | kk) != 0 ? 1u : 0u);
      ptx::mma_commit(&empty[s]);
    }
    ptx::mma_commit(done);
  }
  __syncwarp();
  const bool ok = ptx::mbar_wait(done, 0);
  ptx::tc_fence_after();
  if (!ok && tid == 0) {
    flags[0] = 1;
    latch_error(ctrl, kErrTimeout, 402);
  }
  __syncthreads();
  ptx::grid_dep_launch();
  if (!flags[0]) {
    const int r = warp * 32 + lane, m = xrow0 + r;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    const int n0 = ft * kBN;
    const int b = m / ep.C, i = m % ep.C, pos = ep.p0 + i;
    const bool valid = ep.gblk ? true : m < ep.Mc;  // packed expert blocks: padding rows are computed, never read
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      float lo[16], hi[16];
      ptx::tmem_ld16(trow + 16 * c, lo);       // features n0 + 16c + q
      ptx::tmem_ld16(trow + 64 + 16 * c, hi);  // features n0 + 64 + 16c + q
      if (!valid) continue;
      if (ep.op == BP_QKV) {
        if (n0 < ep.qdim + ep.kvdim) {
          // rotate-half RoPE of pair (j, j + 64) at this row's position
          const float* cs = ep.rope + (size_t)pos * kHD;
          float ra[16], rb[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int j = 16 * c + q;
            const float cv = cs[2 * j], sv = cs[2 * j + 1];
            ra[q] = lo[q] * cv - hi[q] * sv;
            rb[q] = hi[q] * cv + lo[q] * sv;
          }
          if (n0 < ep.qdim) {
            __nv_bfloat16* qr = ep.q + (size_t)m * ep.qdim + n0;
            store16(qr + 16 * c, ra);
            store16(qr + 64 + 16 * c, rb);
          } else {
            const int g = (n0 - ep.qdim) / kHD, sq = ep.slot0 + b;
            __nv_bfloat16* K =
                ep.kv + kv_index(ep.km, ep.Hkv, kHD, ep.layer, 0, kv_page(ep.km, sq, pos), g, kv_off(ep.km, pos));
            store16(K + 16 * c, ra);
            store16(K + 64 + 16 * c, rb);
          }
        } else {
          const int g = (n0 - ep.qdim - ep.kvdim) / kHD, sq = ep.slot0 + b;
          __nv_bfloat16* V =
              ep.kv + kv_index(ep.km, ep.Hkv, kHD, ep.layer, 1, kv_page(ep.km, sq, pos), g, kv_off(ep.km, pos));
          store16(V + 16 * c, lo);
          store16(V + 64 + 16 * c, hi);
        }
      } else if (ep.op == BP_RESID) {
        float* hr = ep.h + (size_t)m * ep.d + n0;
        add16(hr + 16 * c, lo);
        add16(hr + 64 + 16 * c, hi);
      } else if (ep.op == BP_YOUT) {
        float* yr = ep.y + (size_t)m * ep.ldy + n0;
        float4* y4 = reinterpret_cast<float4*>(yr + 16 * c);
        float4* y5 = reinterpret_cast<float4*>(yr + 64 + 16 * c);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          y4[q] = make_float4(lo[4 * q], lo[4 * q + 1], lo[4 * q + 2], lo[4 * q + 3]);
          y5[q] = make_float4(hi[4 * q], hi[4 * q + 1], hi[4 * q + 2], hi[4 * q + 3]);
        }
      } else {  // BP_SWIGLU: rows 0..63 of the tile are gate, 64..127 up, of z features 64 ft ..
        float zv[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) zv[q] = silu_f(lo[q]) * hi[q];
        store16(ep.z + (size_t)m * ep.F + ft * 64 + 16 * c, zv);
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tmem, kBN);
}

size_t gemm_smem() { return 1024 + (size_t)kStages * kStage + (2 * kStages + 1) * 8 + 16; }

// ------------------------------------------------------------------ causal attention

constexpr int TP = 64;
constexpr int BOX = TP * 64 * 2;   // 64 positions x 64 dims bf16 = 8 KB
constexpr int ASTAGE = 4 * BOX;    // K lo, K hi, V lo, V hi
constexpr int ANS = 2;
constexpr float kScale = 0.08838834764831845f;  // 1/sqrt(128)

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// p = hi + lo with hi = bf16(p), lo = bf16(p - hi), packed in pairs.
__device__ __forceinline__ void split_pair(float x, float y, uint32_t& hi, uint32_t& lo) {
  __nv_bfloat162 hv = __floats2bfloat162_rn(x, y);
  float2 hf = __bfloat1622float2(hv);
  hi = *reinterpret_cast<uint32_t*>(&hv);
  lo = pack2(x - hf.x, y - hf.y);
}

__device__ __forceinline__ uint32_t sw_off(int pos, int dim) {
  const int box = dim >> 6, dd = dim & 63;
  return box * BOX + pos * 128 + ((((dd >> 3) ^ (pos & 7)) << 4)) + ((dd & 7) << 1);
}

// Grid (64-query block, query head, sequence).  Chunk rows are sequence-major:
// row b*C + i holds position p0 + i of sequence b.
__global__ void __launch_bounds__(160, 1)
    k_bp_attn(const __grid_constant__ CUtensorMap tkv, const __nv_bfloat16* __restrict__ q,
              __nv_bfloat16* __restrict__ o, Ctrl* __restrict__ ctrl, int layer, KvMap km, int slot0, int Hkv,
              int G, int qdim, int C, int p0) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + ANS * ASTAGE);
  uint64_t* empty = full + ANS;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + ANS);
  const int qb = blockIdx.x, h = blockIdx.y, b = blockIdx.z, g = h / G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i0 = qb * TP;
  const int nq = min(TP, C - i0);
  const int kend = p0 + i0 + nq;  // keys [0, kend): the cache up to the block's last query
  const int ntiles = (kend + TP - 1) / TP;
  // tensor-map rows of the K / V blocks of the page holding key position p
  // (a 64-position tile never spans two pages), and its offset there
  const int sq = slot0 + b;
  auto tile_z = [&](int p, int kvsel) { return ((layer * 2 + kvsel) * km.NP + kv_page(km, sq, p)) * Hkv + g; };
  if (tid == 0) {
    for (int i = 0; i < ANS; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&empty[i], 4);
    }
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
  }
  __syncthreads();
  ptx::grid_dep_wait();  // the queries and this chunk's K/V come from the QKV GEMM
  ptx::grid_dep_launch();

  if (warp == 4) {
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % ANS;
        if (i >= ANS && !ptx::mbar_wait(&empty[st], ((i / ANS) - 1) & 1)) {
          *abort_flag = 1;
          latch_error(ctrl, kErrTimeout, 410);
          break;
        }
        if (*abort_flag) break;
        const int kp = i * TP, zK = tile_z(kp, 0), zV = tile_z(kp, 1), y = kv_off(km, kp);
        uint8_t* dst = ring + st * ASTAGE;
        ptx::mbar_arrive_expect_tx(&full[st], ASTAGE);
        ptx::tma_load_3d(dst + 0 * BOX, &tkv, &full[st], 0, y, zK);
        ptx::tma_load_3d(dst + 1 * BOX, &tkv, &full[st], 64, y, zK);
        ptx::tma_load_3d(dst + 2 * BOX, &tkv, &full[st], 0, y, zV);
        ptx::tma_load_3d(dst + 3 * BOX, &tkv, &full[st], 64, y, zV);
        issued = i + 1;
      }
      if (*abort_flag)
        for (int i = issued - ANS < 0 ? 0 : issued - ANS; i < issued; ++i)
          ptx::mbar_wait(&full[i % ANS], (i / ANS) & 1, 100000000ull);
    }
    return;
  }

  // ---- compute warps: queries i0 + 16 warp + {gq, gq + 8}
  const int gq = lane >> 2, tq = lane & 3, mq = lane >> 3, r8 = lane & 7;
  const int iq0 = i0 + warp * 16 + gq, iq1 = iq0 + 8;
  const int qp0 = p0 + iq0, qp1 = p0 + iq1;  // absolute positions
  const bool v0 = iq0 < C, v1 = iq1 < C;
  uint32_t qa[8][4];
  {
    const __nv_bfloat16* q0 = q + (size_t)(b * C + (v0 ? iq0 : 0)) * qdim + h * kHD;
    const __nv_bfloat16* q1 = q + (size_t)(b * C + (v1 ? iq1 : 0)) * qdim + h * kHD;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      qa[kk][0] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + kk * 16 + 2 * tq) : 0u;
      qa[kk][1] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + kk * 16 + 2 * tq) : 0u;
      qa[kk][2] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + kk * 16 + 8 + 2 * tq) : 0u;
      qa[kk][3] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + kk * 16 + 8 + 2 * tq) : 0u;
    }
  }
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  float oacc[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;

  for (int it = 0; it < ntiles; ++it) {
    const int st = it % ANS;
    const bool okw = __all_sync(0xffffffffu, ptx::mbar_wait(&full[st], (it / ANS) & 1));
    if (!okw) {
      if (lane == 0) {
        *abort_flag = 1;
        latch_error(ctrl, kErrTimeout, 411);
      }
      break;
    }
    if (*abort_flag) break;
    const uint32_t kbase = ptx::smem_u32(ring + st * ASTAGE);
    const uint32_t vbase = kbase + 2 * BOX;
    // S[16 queries][64 keys]: n-tile nt = keys 8 nt .. 8 nt + 7
    float sc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b00, b01, b10, b11;
        ldsm_x4(kbase + sw_off(16 * np + (mq >> 1) * 8 + r8, kk * 16 + (mq & 1) * 8), b00, b01, b10, b11);
        mma_16816(sc[2 * np], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b00, b01);
        mma_16816(sc[2 * np + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b10, b11);
      }
    }
    // causal mask, online softmax for rows gq (elements 0, 1) and gq + 8 (2, 3)
    const int kbase_pos = it * TP + 2 * tq;
    float corr[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int qp = hh ? qp1 : qp0;
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kp = kbase_pos + nt * 8 + e;
          const float v = kp <= qp ? sc[nt][2 * hh + e] * kScale : -INFINITY;
          sc[nt][2 * hh + e] = v;
          mx = fmaxf(mx, v);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float mo = m_run[hh], mn = fmaxf(mo, mx);
      corr[hh] = (mo == -INFINITY) ? 0.f : expf(mo - mn);
      float sum = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float v = sc[nt][2 * hh + e];
          const float p = (v == -INFINITY) ? 0.f : expf(v - mn);
          sc[nt][2 * hh + e] = p;
          sum += p;
        }
      m_run[hh] = mn;
      l_run[hh] = l_run[hh] * corr[hh] + sum;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      oacc[j][0] *= corr[0];
      oacc[j][1] *= corr[0];
      oacc[j][2] *= corr[1];
      oacc[j][3] *= corr[1];
    }
    // O += P V over four 16-key chunks
#pragma unroll
    for (int kc = 0; kc < 4; ++kc) {
      uint32_t ph[4], pl[4];
      split_pair(sc[2 * kc][0], sc[2 * kc][1], ph[0], pl[0]);
      split_pair(sc[2 * kc][2], sc[2 * kc][3], ph[1], pl[1]);
      split_pair(sc[2 * kc + 1][0], sc[2 * kc + 1][1], ph[2], pl[2]);
      split_pair(sc[2 * kc + 1][2], sc[2 * kc + 1][3], ph[3], pl[3]);
#pragma unroll
      for (int j2 = 0; j2 < 8; ++j2) {
        uint32_t w00, w01, w10, w11;
        ldsm_x4_t(vbase + sw_off(16 * kc + (mq & 1) * 8 + r8, j2 * 16 + (mq >> 1) * 8), w00, w01, w10, w11);
        mma_16816(oacc[2 * j2], ph[0], ph[1], ph[2], ph[3], w00, w01);
        mma_16816(oacc[2 * j2], pl[0], pl[1], pl[2], pl[3], w00, w01);
        mma_16816(oacc[2 * j2 + 1], ph[0], ph[1], ph[2], ph[3], w10, w11);
        mma_16816(oacc[2 * j2 + 1], pl[0], pl[1], pl[2], pl[3], w10, w11);
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&empty[st]);
  }
  if (*abort_flag) return;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 1);
    l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 2);
  }
  const float inv0 = 1.f / l_run[0], inv1 = 1.f / l_run[1];
  __nv_bfloat16* o0 = o + (size_t)(b * C + iq0) * qdim + h * kHD;
  __nv_bfloat16* o1 = o + (size_t)(b * C + iq1) * qdim + h * kHD;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int dcol = j * 8 + 2 * tq;
    if (v0) *reinterpret_cast<uint32_t*>(o0 + dcol) = pack2(oacc[j][0] * inv0, oacc[j][1] * inv0);
    if (v1) *reinterpret_cast<uint32_t*>(o1 + dcol) = pack2(oacc[j][2] * inv1, oacc[j][3] * inv1);
  }
}

size_t attn_smem() { return 1024 + (size_t)ANS * ASTAGE + 2 * ANS * 8 + 16; }

// ------------------------------------------------------------------ MoE (router replay's primary routing)
//
// "Mecanismos Clave" (Replay de Router): prefill runs the primary flow, whose
// router picks each token's top-k experts (descending router logit, ties to
// the lower index) and gates them with the softmax of those logits.  The
// chunk's rows are grouped by expert: each chosen (row, j) takes a slot in
// its expert's list, the expert's rows are packed into 128-row blocks, the
// expert GEMMs run over the blocks, and each row sums its k gated expert
// outputs in j order.  A row's result does not depend on its slot, so the
// order in which rows take slots does not change any value.

constexpr int kRouteWarps = 8;
constexpr int kMaxRouteK = 16;

__global__ void __launch_bounds__(32 * kRouteWarps)
    k_pf_route(const float* __restrict__ rlog, int Mc, int E, int k, int* __restrict__ ecount,
               int* __restrict__ sel_e, int* __restrict__ sel_slot, float* __restrict__ sel_g) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  __shared__ int ch[kRouteWarps][kMaxRouteK];
  __shared__ float cv[kRouteWarps][kMaxRouteK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = blockIdx.x * kRouteWarps + warp;
  if (m >= Mc) return;  // uniform across the warp
  const float* r = rlog + (size_t)m * E;
  uint32_t taken = 0;  // bit t: expert lane + 32 t already chosen (E <= 1024)
  for (int j = 0; j < k; ++j) {
    // a NaN logit counts as -inf, and ties go to the lower index, so one of
    // the (at least E - j > 0) untaken experts is always chosen
    float best = -INFINITY;
    int bi = E;
    for (int t = 0, e = lane; e < E; ++t, e += 32) {
      if ((taken >> t) & 1u) continue;
      float v = r[e];
      if (!(v == v)) v = -INFINITY;
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
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == 0) {
      ch[warp][j] = bi;
      cv[warp][j] = best;
    }
  }
  __syncwarp();
  if (lane == 0) {
    // softmax over the chosen logits (the first is the largest)
    float mx = -INFINITY;
    for (int j = 0; j < k; ++j) mx = fmaxf(mx, cv[warp][j]);
    float den = 0.f;
    for (int j = 0; j < k; ++j) den += expf(cv[warp][j] - mx);
    for (int j = 0; j < k; ++j) {
      const int e = ch[warp][j];
      sel_e[(size_t)m * k + j] = e;
      sel_slot[(size_t)m * k + j] = atomicAdd(&ecount[e], 1);
      sel_g[(size_t)m * k + j] = expf(cv[warp][j] - mx) / den;
    }
  }
}

// Packed layout: expert e's rows start at poff[e] (a multiple of 128); the
// block table lists (expert, first row) for each 128-row block, then -1.
__global__ void k_pf_blocks(const int* __restrict__ ecount, int E, int* __restrict__ poff, int* __restrict__ gblk,
                            int maxblk) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  if (threadIdx.x != 0) return;
  int nb = 0;
  for (int e = 0; e < E; ++e) {
    poff[e] = nb * kBM;
    const int eb = (ecount[e] + kBM - 1) / kBM;
    for (int i = 0; i < eb && nb < maxblk; ++i, ++nb) {
      gblk[2 * nb] = e;
      gblk[2 * nb + 1] = nb * kBM;
    }
  }
  for (int i = nb; i < maxblk; ++i) gblk[2 * i] = -1;
}

// Entry (m, j) = row m's j-th expert: copy normed row m into the expert's
// packed block (one warp per entry, 16-byte copies; d is a multiple of 8).
__global__ void k_pf_gather(const __nv_bfloat16* __restrict__ u, const int* __restrict__ sel_e,
                            const int* __restrict__ sel_slot, const int* __restrict__ poff, int nent, int k, int d,
                            __nv_bfloat16* __restrict__ xg) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ent = blockIdx.x * (blockDim.x >> 5) + warp;
  if (ent >= nent) return;
  const int m = ent / k;
  const int row = poff[sel_e[ent]] + sel_slot[ent];
  const uint4* src = reinterpret_cast<const uint4*>(u + (size_t)m * d);
  uint4* dst = reinterpret_cast<uint4*>(xg + (size_t)row * d);
  for (int i = lane; i < d / 8; i += 32) dst[i] = src[i];
}

// h[m] += sum_j g_j * y[packed row of (m, j)], j in order (fp32).
__global__ void k_pf_combine(const float* __restrict__ yp, const int* __restrict__ sel_e,
                             const int* __restrict__ sel_slot, const float* __restrict__ sel_g,
                             const int* __restrict__ poff, int k, int d, float* __restrict__ h) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int m = blockIdx.x;
  __shared__ int rows[kMaxRouteK];
  __shared__ float gs[kMaxRouteK];
  if (threadIdx.x < k) {
    rows[threadIdx.x] = poff[sel_e[(size_t)m * k + threadIdx.x]] + sel_slot[(size_t)m * k + threadIdx.x];
    gs[threadIdx.x] = sel_g[(size_t)m * k + threadIdx.x];
  }
  __syncthreads();
  float4* hr = reinterpret_cast<float4*>(h + (size_t)m * d);
  for (int c = threadIdx.x; c < d / 4; c += blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const float4 y = reinterpret_cast<const float4*>(yp + (size_t)rows[j] * d)[c];
      const float g = gs[j];
      acc.x = fmaf(g, y.x, acc.x);
      acc.y = fmaf(g, y.y, acc.y);
      acc.z = fmaf(g, y.z, acc.z);
      acc.w = fmaf(g, y.w, acc.w);
    }
    float4 x = hr[c];
    x.x += acc.x;
    x.y += acc.y;
    x.z += acc.z;
    x.w += acc.w;
    hr[c] = x;
  }
}

// ------------------------------------------------------------------ embedding

// h[b*C + i] = E1[tokens[b][p0 + i]] for the chunk (primary flow only).
__global__ void k_bp_embed(const __nv_bfloat16* __restrict__ e1, const int32_t* __restrict__ tok, int n, int C,
                           int p0, float* __restrict__ h, int d, int V, Ctrl* ctrl) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int m = blockIdx.x, b = m / C, i = m % C;
  const int id = tok[(size_t)b * n + p0 + i];
  const bool ok = id >= 0 && id < V;
  if (!ok && threadIdx.x == 0) latch_error(ctrl, kErrDevice, 1000 + b);
  const __nv_bfloat16* e = e1 + (size_t)(ok ? id : 0) * d;
  float* out = h + (size_t)m * d;
  for (int k = threadIdx.x; k < d; k += blockDim.x) out[k] = ok ? __bfloat162float(e[k]) : 0.f;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

bool map_rows(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBM};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename... KArgs, typename... Args>
void launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
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

void gemm(const CUtensorMap& tx, const CUtensorMap& tw, int K, int n_out, const BpEp& ep, Ctrl* ctrl,
          cudaStream_t s, int row_tiles = 0) {
  const dim3 grid(row_tiles ? row_tiles : (ep.Mc + kBM - 1) / kBM, n_out / kBN);
  launch_ex(k_bp_gemm, grid, dim3(128), gemm_smem(), s, tx, tw, K / kBK, ep, ctrl);
}

}  // namespace

int bp_rows(const Dims& D) {
  const char* e = getenv("DF_SERIAL_PREFILL");
  if (e && e[0] == '1') return 0;
  if (!D.bf16 || D.hd != kHD) return 0;
  if (D.d % kBN || D.qdim % kBN || D.kvdim % kBN || D.F % 64 || D.d % kBK || D.qdim % kBK) return 0;
  if (D.E && (D.Fe % 64 || D.E > 1024 || D.k > kMaxRouteK)) return 0;
  if (2 * D.G > 64) return 0;
  const int rows = std::max(kChunkRows, (D.maxB + kBM - 1) / kBM * kBM);
  return rows;
}

// 128-row blocks of the packed expert buffers for chunks of R rows: every
// entry, plus a partial block per expert.
int moe_blocks(const Dims& D, int R) { return (R * D.k + kBM - 1) / kBM + D.E; }

size_t bp_workspace_bytes(const Dims& D) {
  const size_t R = (size_t)bp_rows(D);
  if (!R) return 0;
  size_t b = R * D.d * 4 + R * D.d * 2 + 2 * R * D.qdim * 2 + R * (size_t)D.F * 2 + 5 * 256;
  if (D.E) {
    const size_t rows = (size_t)moe_blocks(D, (int)R) * kBM;
    b += R * D.d * 4 + R * D.E * 4 + 3 * R * D.k * 4 + 2 * (size_t)D.E * 4 + (size_t)moe_blocks(D, (int)R) * 8 +
         rows * D.d * 2 + rows * D.Fe * 2 + rows * D.d * 4 + 12 * 256;
  }
  return b;
}

bool bp_init(BpPlan& P, const Dims& D, void* region, std::string* err) {
  P = BpPlan{};
  const int R = bp_rows(D);
  if (!R || !region || !encode_fn()) return true;
  char* c = static_cast<char*>(region);
  auto take = [&](size_t bytes) {
    char* p = c;
    c += (bytes + 255) / 256 * 256;
    return p;
  };
  P.mcap = R;
  P.h = reinterpret_cast<float*>(take((size_t)R * D.d * 4));
  P.u = take((size_t)R * D.d * 2);
  P.q = take((size_t)R * D.qdim * 2);
  P.o = take((size_t)R * D.qdim * 2);
  P.z = take((size_t)R * (D.F ? D.F : 64) * 2);
  bool ok = map_rows(&P.x_u, P.u, D.d, R) && map_rows(&P.x_o, P.o, D.qdim, R);
  if (D.F) ok = ok && map_rows(&P.x_z, P.z, D.F, R);
  if (D.E) {
    P.moe = true;
    P.maxblk = moe_blocks(D, R);
    const size_t rows = (size_t)P.maxblk * kBM;
    P.un = reinterpret_cast<float*>(take((size_t)R * D.d * 4));
    P.rlog = reinterpret_cast<float*>(take((size_t)R * D.E * 4));
    P.sel_e = reinterpret_cast<int*>(take((size_t)R * D.k * 4));
    P.sel_slot = reinterpret_cast<int*>(take((size_t)R * D.k * 4));
    P.sel_g = reinterpret_cast<float*>(take((size_t)R * D.k * 4));
    P.ecount = reinterpret_cast<int*>(take((size_t)D.E * 4));
    P.poff = reinterpret_cast<int*>(take((size_t)D.E * 4));
    P.gblk = reinterpret_cast<int*>(take((size_t)P.maxblk * 8));
    P.xg = take(rows * D.d * 2);
    P.zg = take(rows * D.Fe * 2);
    P.yg = reinterpret_cast<float*>(take(rows * D.d * 4));
    ok = ok && map_rows(&P.x_xg, P.xg, D.d, rows) && map_rows(&P.x_zg, P.zg, D.Fe, rows);
  }
  if (!ok) {
    if (err) *err = "cuTensorMapEncodeTiled failed (prefill activation maps)";
    return false;
  }
  if (cudaFuncSetAttribute(k_bp_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gemm_smem()) != cudaSuccess ||
      cudaFuncSetAttribute(k_bp_attn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)attn_smem()) !=
          cudaSuccess) {
    cudaGetLastError();
    return true;  // stays disabled
  }
  P.enabled = true;
  return true;
}

void bp_prefill(const BpPlan& P, const TcPlan& tc, const AttnPlan& at, const MoePlan* moe, const Dims& D,
                const Buffers& Bf, void* kv, const void* emb1, const float* const* attn_norm,
                const float* const* mlp_norm, const void* const* router, const int32_t* tokens, int B, int n,
                int slot0, cudaStream_t s) {
  const int C = std::max(1, P.mcap / B);
  __nv_bfloat16* kvb = static_cast<__nv_bfloat16*>(kv);
  for (int p0 = 0; p0 < n; p0 += C) {
    const int Ce = std::min(C, n - p0), Mc = B * Ce;
    launch_ex(k_bp_embed, dim3(Mc), dim3(256), 0, s, static_cast<const __nv_bfloat16*>(emb1), tokens, n, Ce, p0,
              P.h, D.d, D.V, Bf.ctrl);
    BpEp ep{};
    ep.Mc = Mc;
    ep.C = Ce;
    ep.p0 = p0;
    ep.q = static_cast<__nv_bfloat16*>(P.q);
    ep.qdim = D.qdim;
    ep.kvdim = D.kvdim;
    ep.Hkv = D.Hkv;
    ep.kv = kvb;
    ep.km = Bf.kvm;
    ep.slot0 = slot0;
    ep.rope = Bf.rope;
    ep.h = P.h;
    ep.d = D.d;
    ep.z = static_cast<__nv_bfloat16*>(P.z);
    ep.F = D.F;
    for (int l = 0; l < D.L; ++l) {
      ep.layer = l;
      launch_rmsnorm_rows(D, P.h, attn_norm[l], P.u, Mc, s);
      ep.op = BP_QKV;
      gemm(P.x_u, tc.w_qkv[l], D.d, D.qkvn, ep, Bf.ctrl, s);
      launch_ex(k_bp_attn, dim3((Ce + TP - 1) / TP, D.Hq, B), dim3(160), attn_smem(), s, at.kv,
                static_cast<const __nv_bfloat16*>(P.q), static_cast<__nv_bfloat16*>(P.o), Bf.ctrl, l, Bf.kvm, slot0,
                D.Hkv, D.G, D.qdim, Ce, p0);
      ep.op = BP_RESID;
      gemm(P.x_o, tc.w_o[l], D.qdim, D.d, ep, Bf.ctrl, s);
      if (!D.E) {
        launch_rmsnorm_rows(D, P.h, mlp_norm[l], P.u, Mc, s);
        ep.op = BP_SWIGLU;
        gemm(P.x_u, tc.w_gu[l], D.d, 2 * D.F, ep, Bf.ctrl, s);
        ep.op = BP_RESID;
        gemm(P.x_z, tc.w_d[l], D.F, D.d, ep, Bf.ctrl, s);
        continue;
      }
      // MoE layer: route the chunk's rows, run the experts over their packed
      // blocks, add each row's gated expert outputs to its residual
      launch_rmsnorm_rows(D, P.h, mlp_norm[l], P.u, Mc, s, P.un);
      launch_router_rows(D, router[l], P.un, P.rlog, Mc, s);
      cudaMemsetAsync(P.ecount, 0, (size_t)D.E * 4, s);
      launch_ex(k_pf_route, dim3((Mc + kRouteWarps - 1) / kRouteWarps), dim3(32 * kRouteWarps), 0, s,
                (const float*)P.rlog, Mc, D.E, D.k, P.ecount, P.sel_e, P.sel_slot, P.sel_g);
      launch_ex(k_pf_blocks, dim3(1), dim3(32), 0, s, (const int*)P.ecount, D.E, P.poff, P.gblk, P.maxblk);
      const int nent = Mc * D.k;
      launch_ex(k_pf_gather, dim3((nent + 7) / 8), dim3(256), 0, s, static_cast<const __nv_bfloat16*>(P.u),
                (const int*)P.sel_e, (const int*)P.sel_slot, (const int*)P.poff, nent, D.k, D.d,
                static_cast<__nv_bfloat16*>(P.xg));
      BpEp eg = ep;
      eg.gblk = P.gblk;
      eg.op = BP_SWIGLU;
      eg.z = static_cast<__nv_bfloat16*>(P.zg);
      eg.F = D.Fe;
      eg.wrows = 2 * D.Fe;
      gemm(P.x_xg, moe->w_gu[l], D.d, 2 * D.Fe, eg, Bf.ctrl, s, P.maxblk);
      eg.op = BP_YOUT;
      eg.y = P.yg;
      eg.ldy = D.d;
      eg.wrows = D.d;
      gemm(P.x_zg, moe->w_d[l], D.Fe, D.d, eg, Bf.ctrl, s, P.maxblk);
      launch_ex(k_pf_combine, dim3(Mc), dim3(256), 0, s, (const float*)P.yg, (const int*)P.sel_e,
                (const int*)P.sel_slot, (const float*)P.sel_g, (const int*)P.poff, D.k, D.d, P.h);
    }
  }
}

}  // namespace df
