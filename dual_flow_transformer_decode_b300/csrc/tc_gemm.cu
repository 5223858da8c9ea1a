// Swap-AB tensor-core GEMM for the stacked-row projections of the decode
// step, with the step's epilogues fused:
//
//   D^T[128 weight rows][N stacked rows] = W_tile[128][K] · X[N][K]^T
//
// W (the shared weight matrix) is the MMA "A" operand, 128 rows per tile,
// K-major; X (the stacked primary + auxiliary rows, padded to N, a multiple
// of 16) is the "B" operand.  Both are staged by TMA in the 128-byte-swizzled
// layout through an mbarrier ring; one elected thread issues tcgen05.mma
// (kind::f16, bf16 inputs, fp32 accumulate) into a TMEM accumulator of N
// columns; four warps drain it with tcgen05.ld.  Every weight byte is read
// once per step for both flows ("Mecanismos Clave": grouped execution loads
// the weights once for both flows).
//
// Split-K: the K-splits of one tile form a thread-block cluster (up to 16
// CTAs).  Each CTA leaves its partial tile in shared memory; after a cluster
// barrier CTA r sums slice r of the tile over all ranks through distributed
// shared memory, in rank order, and runs the epilogue on that slice.  The
// split count targets two resident CTAs per SM (one CTA streams ~35 GB/s,
// so a single CTA per SM cannot saturate HBM).  Results are deterministic,
// and each column (stacked row) depends only on its own inputs, so the
// primary rows are bit-identical whether or not the auxiliary rows are
// present.  The first ring stages' weight tiles are requested before
// griddepcontrol.wait (weights do not depend on the previous kernel), and
// the epilogue's parameters (coupling-vector slice, RoPE row) are staged in
// shared memory by the otherwise idle warps during the main loop.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cooperative_groups.h>
#include <cstdio>
#include <cstdlib>

#include "ptx.cuh"
#include "tc_gemm.h"

namespace df {

namespace cg = cooperative_groups;

namespace {

constexpr int kMaxStages = 8;
#ifndef DF_GEMM_WIDE_KB
#define DF_GEMM_WIDE_KB 96
#endif
constexpr int kBK = 64;                 // K elements per stage (one 128-byte swizzle atom of bf16)
constexpr int kBM = 128;                // weight rows per tile (MMA M)
constexpr int kStageW = kBM * kBK * 2;  // 16 KB
constexpr int kMaxSplit = 16;           // largest cluster (non-portable size)
constexpr int kStP = kBM + 4;           // row stride (floats) of the partial tile: rows 4 banks apart
constexpr int kWideN = 128;             // above this many stacked rows a tile takes a whole SM
constexpr int kWideKB = 200;            // ring budget of such a tile (the partial tile reuses it)

struct EpArgs {
  int op;
  // Failure-detection test hook (0 in normal use): the producer first waits
  // this many nanoseconds on a barrier nothing arrives on, lets that bounded
  // wait run out, latches the timeout and issues no copy.
  unsigned long long stall_ns;
  int lo, hi, B;  // active stacked rows
  int n_out;      // valid output features of the matrix
  // QKV
  const float* a;
  __nv_bfloat16* kv;   // the cache (all layers)
  int layer;
  KvMap km;            // cache addressing; paged mode: per-sequence positions
  const float* rope;
  const Ctrl* ctrl;
  float* qatt;
  int qdim, kvdim, hd, Hkv;
  // couplings
  Couple C;
  const float* bvec;
  const float* cvec;
  // outputs
  float* h;
  int d;
  __nv_bfloat16* z;
  int F;
  float* logits;
  int V;
  // wide tiles with split-K: partial tiles in global memory (L2), one
  // [N][kStP] tile per (tile, split) of the launch
  float* gpart;
};

// Reduced values of one (row, quad) unit: features p..p+3 and p+64..p+67 of
// the tile (p a multiple of 4), i.e. four (p, p + 64) pairs.
struct Quad {
  float4 lo, hi;
};

__device__ __forceinline__ float4 f4add(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}
__device__ __forceinline__ float f4get(const float4& v, int k) { return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w; }
__device__ __forceinline__ void f4set(float4& v, int k, float x) {
  if (k == 0) v.x = x;
  else if (k == 1) v.y = x;
  else if (k == 2) v.z = x;
  else v.w = x;
}

// Sums of the cluster's partial tiles for rows m1 and m2 (each if its flag
// is set), features p..p+3 and p+64..p+67, in cluster-rank (K-split) order,
// element by element (the same order for every element as a scalar sum).
// The partial tiles are the ranks' shared memory (distributed shared
// memory), or, with gp set, the ranks' tiles in global memory at gp +
// rank * gstride.  Loads are issued four ranks at a time for both rows
// before they are added.
__device__ __forceinline__ void reduce_quads(cg::cluster_group& cl, float* st, int S, int m1, bool has1, int m2,
                                             bool has2, int p, Quad& q1, Quad& q2, const float* gp, size_t gstride) {
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  q1 = Quad{z, z};
  q2 = Quad{z, z};
  if (S == 1) {
    if (has1)
      q1 = Quad{*reinterpret_cast<const float4*>(st + m1 * kStP + p),
                *reinterpret_cast<const float4*>(st + m1 * kStP + p + 64)};
    if (has2)
      q2 = Quad{*reinterpret_cast<const float4*>(st + m2 * kStP + p),
                *reinterpret_cast<const float4*>(st + m2 * kStP + p + 64)};
    return;
  }
  for (int s0 = 0; s0 < S; s0 += 4) {
    float4 a[4], b[4], c[4], d[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (s0 + j < S) {
        const float* r = gp ? gp + (size_t)(s0 + j) * gstride : cl.map_shared_rank(st, s0 + j);
        if (has1) {
          a[j] = *reinterpret_cast<const float4*>(r + m1 * kStP + p);
          b[j] = *reinterpret_cast<const float4*>(r + m1 * kStP + p + 64);
        }
        if (has2) {
          c[j] = *reinterpret_cast<const float4*>(r + m2 * kStP + p);
          d[j] = *reinterpret_cast<const float4*>(r + m2 * kStP + p + 64);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (s0 + j < S) {
        if (has1) {
          q1.lo = f4add(q1.lo, a[j]);
          q1.hi = f4add(q1.hi, b[j]);
        }
        if (has2) {
          q2.lo = f4add(q2.lo, c[j]);
          q2.hi = f4add(q2.hi, d[j]);
        }
      }
    }
  }
}

// SiLU with the fast exponential and division: the product feeds a bf16
// rounding, far coarser than their few-ulp error.
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

__device__ __forceinline__ uint2 pack4_bf16(float a, float b, float c, float d) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
  return make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
}

// Epilogue parameters of pairs [p0, p1), staged in shared memory:
//   par[0][pp], par[1][pp]  RoPE cos/sin of pair p0+pp at position t (QKV)
//   par[2][pp], par[3][pp]  coupling vector at features p, p+64 (a for Q
//                           tiles, b for SwiGLU tiles, c for down tiles)
__device__ __forceinline__ void stage_params(const EpArgs& ep, float* par, int n0, int p0, int np, int i) {
  if (i >= np) return;
  const int p = p0 + i, g0 = n0 + p, g1 = g0 + 64;
  float c = 0.f, s = 0.f, x = 0.f, y = 0.f;
  switch (ep.op) {
    case (int)TcOp::QKV: {
      const float* cs = ep.rope + (size_t)ep.ctrl->t * ep.hd;
      c = cs[2 * p];
      s = cs[2 * p + 1];
      if (n0 < ep.qdim) {
        x = ep.a[g0];
        y = ep.a[g1];
      }
      break;
    }
    case (int)TcOp::SWIGLU:
      x = ep.bvec[(n0 / kBM) * 64 + p];
      break;
    case (int)TcOp::DOWN:
      if (g0 < ep.n_out) x = ep.cvec[g0];
      if (g1 < ep.n_out) y = ep.cvec[g1];
      break;
    default:
      break;
  }
  par[0 * 64 + i] = c;
  par[1 * 64 + i] = s;
  par[2 * 64 + i] = x;
  par[3 * 64 + i] = y;
}

// Epilogue over the pairs [p0, p1) (multiples of 4) of a 128-row weight tile
// starting at output feature n0.  Work unit: (sequence b, quad of pairs);
// the unit handles the primary row b and the auxiliary row B+b together, so
// the coupling partner of an auxiliary row is at hand.  Features p and p+64
// form a RoPE pair (head_dim 128) or a gate/up pair (SwiGLU tiles interleave
// 64 gate and 64 up rows).  Shared, global and cache accesses of a unit are
// 16-byte (fp32) or 8-byte (bf16) vectors of its four consecutive features.
__device__ __forceinline__ void epilogue(const EpArgs& ep, cg::cluster_group& cl, float* st, const float* par,
                                         int S, int n0, int p0, int p1, int tid, int nthreads, const float* gp,
                                         size_t gstride) {
  const int nq = (p1 - p0) >> 2;
  const bool prim = ep.lo < ep.B, aux = ep.hi > ep.B;
  const int B = ep.B;
  // paged mode: every sequence at its own position, so the RoPE angles are
  // read per unit instead of from the staged table
  const bool ragged = ep.km.table != nullptr;
  const int t = ep.op == (int)TcOp::QKV && !ragged ? ep.ctrl->t : 0;
  // thread -> unit: consecutive threads take consecutive quads of one row
  // (contiguous row segments in the partial tiles and in the outputs)
  for (int u = tid; u < B * nq; u += nthreads) {
    const int b = u / nq, pp = (u % nq) << 2, p = p0 + pp;
    Quad v1, v2;
    reduce_quads(cl, st, S, b, prim, B + b, aux, p, v1, v2, gp, gstride);
    const int g0 = n0 + p, g1 = n0 + p + 64;
    float4 c = *reinterpret_cast<const float4*>(par + pp), sn = *reinterpret_cast<const float4*>(par + 64 + pp);
    const float4 cx = *reinterpret_cast<const float4*>(par + 128 + pp);
    const float4 cy = *reinterpret_cast<const float4*>(par + 192 + pp);
    switch (ep.op) {
      case (int)TcOp::QKV: {
        int tb = t;
        if (ragged) {
          tb = ep.km.pos[b];
          const float4* cs = reinterpret_cast<const float4*>(ep.rope + (size_t)tb * ep.hd + 2 * p);
          const float4 c01 = cs[0], c23 = cs[1];  // (cos, sin) of pairs p..p+3
          c = make_float4(c01.x, c01.z, c23.x, c23.z);
          sn = make_float4(c01.y, c01.w, c23.y, c23.w);
        }
        if (n0 < ep.qdim) {
          if (prim) {
            if (ep.C.save) {
              *reinterpret_cast<float4*>(ep.C.q1s + (size_t)b * ep.qdim + g0) = v1.lo;
              *reinterpret_cast<float4*>(ep.C.q1s + (size_t)b * ep.qdim + g1) = v1.hi;
            }
            float4 r0, r1;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float lo = f4get(v1.lo, k), hi = f4get(v1.hi, k), ck = f4get(c, k), sk = f4get(sn, k);
              f4set(r0, k, Num<__nv_bfloat16>::quant(lo * ck - hi * sk));
              f4set(r1, k, Num<__nv_bfloat16>::quant(hi * ck + lo * sk));
            }
            *reinterpret_cast<float4*>(ep.qatt + (size_t)b * ep.qdim + g0) = r0;
            *reinterpret_cast<float4*>(ep.qatt + (size_t)b * ep.qdim + g1) = r1;
          }
          if (aux) {
            float4 q0 = v1.lo, q1 = v1.hi;
            if (ep.C.saved) {
              q0 = *reinterpret_cast<const float4*>(ep.C.q1s + (size_t)b * ep.qdim + g0);
              q1 = *reinterpret_cast<const float4*>(ep.C.q1s + (size_t)b * ep.qdim + g1);
            }
            float4 r0, r1;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float a0 = fmaf(f4get(cx, k), f4get(q0, k), f4get(v2.lo, k));
              const float a1 = fmaf(f4get(cy, k), f4get(q1, k), f4get(v2.hi, k));
              const float ck = f4get(c, k), sk = f4get(sn, k);
              f4set(r0, k, Num<__nv_bfloat16>::quant(a0 * ck - a1 * sk));
              f4set(r1, k, Num<__nv_bfloat16>::quant(a1 * ck + a0 * sk));
            }
            const size_t m = (size_t)(B + b) * ep.qdim;
            *reinterpret_cast<float4*>(ep.qatt + m + g0) = r0;
            *reinterpret_cast<float4*>(ep.qatt + m + g1) = r1;
          }
        } else if (prim) {
          const bool isk = n0 < ep.qdim + ep.kvdim;
          const int g = (isk ? n0 - ep.qdim : n0 - ep.qdim - ep.kvdim) / ep.hd;
          __nv_bfloat16* P = ep.kv + kv_index(ep.km, ep.Hkv, ep.hd, ep.layer, isk ? 0 : 1, kv_page(ep.km, b, tb), g,
                                              kv_off(ep.km, tb));
          float4 r0 = v1.lo, r1 = v1.hi;
          if (isk) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float lo = f4get(v1.lo, k), hi = f4get(v1.hi, k), ck = f4get(c, k), sk = f4get(sn, k);
              f4set(r0, k, lo * ck - hi * sk);
              f4set(r1, k, hi * ck + lo * sk);
            }
          }
          *reinterpret_cast<uint2*>(P + p) = pack4_bf16(r0.x, r0.y, r0.z, r0.w);
          *reinterpret_cast<uint2*>(P + p + 64) = pack4_bf16(r1.x, r1.y, r1.z, r1.w);
        }
        break;
      }
      case (int)TcOp::RESID: {
        // every residual value this unit updates is loaded before any store
        // (n_out is a multiple of the tile: all four features are valid)
        float4* h1 = reinterpret_cast<float4*>(ep.h + (size_t)b * ep.d + g0);
        float4* h2 = reinterpret_cast<float4*>(ep.h + (size_t)(B + b) * ep.d + g0);
        const float4 a0 = prim ? h1[0] : float4{}, a1 = prim ? h1[16] : float4{};
        const float4 c0 = aux ? h2[0] : float4{}, c1 = aux ? h2[16] : float4{};
        if (prim) {
          h1[0] = f4add(a0, v1.lo);
          h1[16] = f4add(a1, v1.hi);
        }
        if (aux) {
          h2[0] = f4add(c0, v2.lo);
          h2[16] = f4add(c1, v2.hi);
        }
        break;
      }
      case (int)TcOp::SWIGLU: {
        const int fi = (n0 / kBM) * 64 + p;
        float4 z1;
#pragma unroll
        for (int k = 0; k < 4; ++k) f4set(z1, k, silu_fast(f4get(v1.lo, k)) * f4get(v1.hi, k));
        if (prim) {
          if (ep.C.save) *reinterpret_cast<float4*>(ep.C.z1s + (size_t)b * ep.F + fi) = z1;
          *reinterpret_cast<uint2*>(ep.z + (size_t)b * ep.F + fi) = pack4_bf16(z1.x, z1.y, z1.z, z1.w);
        }
        if (aux) {
          const float4 zp = ep.C.saved ? *reinterpret_cast<const float4*>(ep.C.z1s + (size_t)b * ep.F + fi) : z1;
          float4 z2;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            f4set(z2, k, fmaf(f4get(cx, k), f4get(zp, k), silu_fast(f4get(v2.lo, k)) * f4get(v2.hi, k)));
          *reinterpret_cast<uint2*>(ep.z + (size_t)(B + b) * ep.F + fi) = pack4_bf16(z2.x, z2.y, z2.z, z2.w);
        }
        break;
      }
      case (int)TcOp::DOWN: {
        // loads first (residual values, saved primary outputs), then stores
        float4* h1 = reinterpret_cast<float4*>(ep.h + (size_t)b * ep.d + g0);
        float4* h2 = reinterpret_cast<float4*>(ep.h + (size_t)(B + b) * ep.d + g0);
        const float4* ys = reinterpret_cast<const float4*>(ep.C.y1s + (size_t)b * ep.d + g0);
        const float4 a0 = prim ? h1[0] : float4{}, a1 = prim ? h1[16] : float4{};
        const float4 c0 = aux ? h2[0] : float4{}, c1 = aux ? h2[16] : float4{};
        const bool sv = aux && ep.C.saved;
        const float4 yp0 = sv ? ys[0] : v1.lo, yp1 = sv ? ys[16] : v1.hi;
        if (prim) {
          if (ep.C.save) {
            float4* yw = reinterpret_cast<float4*>(ep.C.y1s + (size_t)b * ep.d + g0);
            yw[0] = v1.lo;
            yw[16] = v1.hi;
          }
          h1[0] = f4add(a0, v1.lo);
          h1[16] = f4add(a1, v1.hi);
        }
        if (aux) {
          float4 r0, r1;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            f4set(r0, k, f4get(c0, k) + fmaf(f4get(cx, k), f4get(yp0, k), f4get(v2.lo, k)));
            f4set(r1, k, f4get(c1, k) + fmaf(f4get(cy, k), f4get(yp1, k), f4get(v2.hi, k)));
          }
          h2[0] = r0;
          h2[16] = r1;
        }
        break;
      }
      case (int)TcOp::LOGITS: {
        if ((ep.V & 3) == 0 && g1 + 3 < ep.n_out) {
          // rows 16-byte aligned and all eight features valid
          if (prim) {
            *reinterpret_cast<float4*>(ep.logits + (size_t)b * ep.V + g0) = v1.lo;
            *reinterpret_cast<float4*>(ep.logits + (size_t)b * ep.V + g1) = v1.hi;
          }
          if (aux) {
            *reinterpret_cast<float4*>(ep.logits + (size_t)(B + b) * ep.V + g0) = v2.lo;
            *reinterpret_cast<float4*>(ep.logits + (size_t)(B + b) * ep.V + g1) = v2.hi;
          }
          break;
        }
        // otherwise (a vocabulary not a multiple of 4, or the last tile)
        // scalar stores, each checked
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (g0 + k < ep.n_out) {
            if (prim) ep.logits[(size_t)b * ep.V + g0 + k] = f4get(v1.lo, k);
            if (aux) ep.logits[(size_t)(B + b) * ep.V + g0 + k] = f4get(v2.lo, k);
          }
          if (g1 + k < ep.n_out) {
            if (prim) ep.logits[(size_t)b * ep.V + g1 + k] = f4get(v1.hi, k);
            if (aux) ep.logits[(size_t)(B + b) * ep.V + g1 + k] = f4get(v2.hi, k);
          }
        }
        break;
      }
    }
  }
}

// One CTA = one K-split of one 128-row weight tile; the K-splits of a tile
// form a thread-block cluster (cluster rank = split index).  NT threads:
// warp 0 TMA producer, warp 1 MMA issuer, all of them drain TMEM and run the
// epilogue (256 when the footprint allows one CTA per SM anyway: wide N).
template <int NT, bool DIRECT = false>
__global__ void __launch_bounds__(NT, 1)
    k_tc_gemm(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tx, int N, int kblocks,
              int kStages, EpArgs ep, Ctrl* ctrl) {
  extern __shared__ uint8_t smem_raw[];
  cg::cluster_group cl = cg::this_cluster();
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int stage_x = N * kBK * 2;
  uint8_t* sw = base;
  uint8_t* sx = base + kStages * kStageW;
  // the epilogue's partial tile [N][128] fp32 reuses the ring; the region is
  // the larger of the two
  size_t region = (size_t)kStages * (kStageW + stage_x);
  if (!DIRECT && (size_t)N * kStP * 4 > region) region = (size_t)N * kStP * 4;
  float* par = reinterpret_cast<float*>(base + region);  // [4][64] epilogue parameters
  uint64_t* full = reinterpret_cast<uint64_t*>(par + 4 * 64);
  uint64_t* empty = full + kMaxStages;
  uint64_t* done = empty + kMaxStages;
  uint64_t* never = done + 1;  // no thread arrives on it (the stall hook's wait)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(never + 1);
  volatile int* flags = reinterpret_cast<volatile int*>(tslot + 1);  // [0] abort
  float* st = reinterpret_cast<float*>(base);                       // [N][kStP] partial tile, reuses the ring

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = (int)cl.num_blocks();
  const int split = (int)cl.block_rank();
  const int tile = blockIdx.x / S;
  const int kb0 = (int)((long long)split * kblocks / S), kb1 = (int)((long long)(split + 1) * kblocks / S);
  const int nk = kb1 - kb0;
  const uint32_t ncols = N <= 32 ? 32 : N <= 64 ? 64 : N <= 128 ? 128 : 256;
  // Split tiles reduce through L2 when the tile is wide (more than 128
  // stacked rows) or has three or more K-splits: pulling the ranks' partial
  // tiles through distributed shared memory then costs more than writing
  // each tile to global memory and reading the shares back (measured at 256
  // rows: epilogue 10 us against 4 us; at 32 rows with 6-8 splits the
  // launch is 1.1-1.4 us shorter).  Two splits keep the cluster exchange.
  float* gtile = (S >= 3 || (S > 1 && N > kWideN)) ? ep.gpart + (size_t)tile * S * N * kStP : nullptr;
  // this rank's share of the tile's 64 (p, p + 64) feature pairs, in quads
  const int p0 = 4 * (split * 16 / S), p1 = 4 * ((split + 1) * 16 / S);

  if (tid == 0) {
    ptx::prefetch_tmap(&tw);
    ptx::prefetch_tmap(&tx);
    for (int s = 0; s < kMaxStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(done, 1);
    ptx::mbar_init(never, 1);
    flags[0] = 0;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 0) {
    ptx::tmem_alloc(tslot, ncols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0 && lane == 0 && ep.stall_ns && !ptx::mbar_wait(never, 0, ep.stall_ns)) {
    // the test hook's wait ran out before any copy was issued: nothing is in
    // flight, the MMA issuer sees the flag and stops waiting
    flags[0] = 1;
    latch_error(ctrl, kErrTimeout, 103);
    ptx::grid_dep_wait();
  } else if (warp == 0 && lane == 0) {
    // TMA producer.  The weights do not depend on the previous kernel, so the
    // first stages' weight tiles are requested before waiting for it.
    const uint64_t pol_w = ptx::policy_evict_first();
    const int pre = nk < kStages ? nk : kStages;
    for (int i = 0; i < pre; ++i) {
      ptx::mbar_arrive_expect_tx(&full[i], kStageW + stage_x);
      ptx::tma_load_2d_hint(sw + i * kStageW, &tw, &full[i], (kb0 + i) * kBK, tile * kBM, pol_w);
    }
    ptx::grid_dep_wait();
    for (int i = 0; i < pre; ++i) ptx::tma_load_2d(sx + i * stage_x, &tx, &full[i], (kb0 + i) * kBK, 0);
    for (int i = pre; i < nk; ++i) {
      const int s = i % kStages;
      if (!ptx::mbar_wait(&empty[s], ((i / kStages) - 1) & 1)) {
        flags[0] = 1;
        latch_error(ctrl, kErrTimeout, 100);
        break;
      }
      ptx::mbar_arrive_expect_tx(&full[s], kStageW + stage_x);
      ptx::tma_load_2d_hint(sw + s * kStageW, &tw, &full[s], (kb0 + i) * kBK, tile * kBM, pol_w);
      ptx::tma_load_2d(sx + s * stage_x, &tx, &full[s], (kb0 + i) * kBK, 0);
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    const uint32_t idesc = ptx::idesc_bf16_f32(kBM, N);
    for (int i = 0; i < nk; ++i) {
      const int s = i % kStages;
      if (!ptx::mbar_wait_abort(&full[s], (i / kStages) & 1, flags)) {
        if (!flags[0]) latch_error(ctrl, kErrTimeout, 101);
        flags[0] = 1;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t a0 = ptx::smem_u32(sw + s * kStageW), b0 = ptx::smem_u32(sx + s * stage_x);
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk)
        ptx::mma_bf16(tmem, ptx::desc_sw128(a0 + kk * 32), ptx::desc_sw128(b0 + kk * 32), idesc,
                      (i | kk) != 0 ? 1u : 0u);
      ptx::mma_commit(&empty[s]);
    }
    ptx::mma_commit(done);
  } else if (warp >= 2) {
    // Epilogue parameters are fixed inputs (and the position t was set by an
    // earlier step), so they are staged before the dependency resolves.
    stage_params(ep, par, tile * kBM, p0, p1 - p0, tid - 64);
    ptx::grid_dep_wait();
  } else {
    ptx::grid_dep_wait();
  }
  __syncwarp();

  const bool ok = ptx::mbar_wait(done, 0);
  ptx::tc_fence_after();
  if (!ok && tid == 0) {
    flags[0] = 1;
    latch_error(ctrl, kErrTimeout, 102);
  }
  __syncthreads();
  const bool aborted = flags[0] != 0;

  if constexpr (DIRECT) {
    // LOGITS from TMEM: lane r of a warp's quarter holds vocabulary entry
    // n0 + 32 (w % 4) + r for the stacked rows of each column chunk; a
    // warp's store of one row is 32 consecutive floats
    ptx::grid_dep_launch();
    if (!aborted) {
      const int quarter = warp & 3, r = quarter * 32 + lane, gv = tile * kBM + r;
      const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
      const bool ok_v = gv < ep.n_out;
      for (int j0 = (warp >> 2) * 16; j0 < N; j0 += 16 * (NT / 128)) {
        float v[16];
        ptx::tmem_ld16(trow + j0, v);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int m = j0 + q;
          if (ok_v && m >= ep.lo && m < ep.hi) ep.logits[(size_t)m * ep.V + gv] = v[q];
        }
      }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, ncols);
    return;
  }

  if (!aborted) {
    // TMEM -> partial tile st[column j][weight row r]; warp w reads TMEM
    // lanes 32 (w % 4) .. +31, warps sharing a lane quarter split the
    // 16-column chunks
    const int quarter = warp & 3, r = quarter * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
    // the tile's destination: this CTA's shared memory, or its slot in the
    // global partials when the split tiles are reduced through L2
    float* dst = gtile ? gtile + (size_t)split * N * kStP : st;
    if (N % 32 == 0) {
      for (int j0 = (warp >> 2) * 32; j0 < N; j0 += 32 * (NT / 128)) {
        float v[32];
        ptx::tmem_ld32(trow + j0, v);
#pragma unroll
        for (int q = 0; q < 32; ++q) dst[(j0 + q) * kStP + r] = v[q];
      }
    } else {
      for (int j0 = (warp >> 2) * 16; j0 < N; j0 += 16 * (NT / 128)) {
        float v[16];
        ptx::tmem_ld16(trow + j0, v);
#pragma unroll
        for (int q = 0; q < 16; ++q) dst[(j0 + q) * kStP + r] = v[q];
      }
    }
  }
  ptx::tc_fence_before();
  // Every CTA of the cluster has its partial tile in shared (or global)
  // memory after this.
  cl.sync();
  ptx::grid_dep_launch();
  if (!aborted) epilogue(ep, cl, st, par, S, tile * kBM, p0, p1, tid, NT, gtile, (size_t)N * kStP);
  // Keep this CTA's shared memory alive until the whole cluster has read it
  // (partials reduced through L2 leave nothing to wait for).
  if (!gtile) cl.sync();
  if (warp == 0) ptx::tmem_dealloc(tmem, ncols);
}

// CUDA-core GEMV for a few stacked rows (2B <= kGemvRows), with the same
// fused epilogues.  At so few rows a projection is a weight stream with a
// handful of multiply-adds per weight, so instead of K-splits (and their
// reduction) the weight matrix is divided finer along its output features:
// one CTA takes 8 feature pairs (p, p + 64) of a 128-row tile over the whole
// K range, i.e. 16 weight rows.  Its 256 threads form 4 row groups (4 weight
// rows each) x 64 K lanes; a K lane streams 16-byte chunks (8 bf16) k = 8c
// for c = lane, lane + 64, ... of its 4 rows, two chunks in flight, and
// multiplies each with the same chunk of every stacked row, so a weight is
// read from HBM once and the activations (a few KB, L1/L2-resident) four
// times per chunk.  Sums: per lane in k order, then a butterfly over the 32
// lanes of a warp, then the two warps of a row group in order -- the same
// order for every output, whatever rows are active.  The first chunks'
// weights are loaded before griddepcontrol.wait.
constexpr int kGemvRows = 8;     // most stacked rows the kernel takes
// Crossover against the tensor-core tile, measured on one B300 (dense ~1B
// model, microseconds per launch, tensor-core / GEMV): 2 stacked rows QKV
// 7.3 / 5.5, Wo 6.5 / 5.0, gate/up 15.4 / 20.0, down 11.5 / 13.9, LM head
// 24.7 / 33.2; 4 rows QKV 7.4 / 7.4, Wo 6.5 / 6.7 and every larger matrix
// slower; 8 rows slower everywhere.  The GEMV therefore takes 2 stacked rows
// (one sequence) and matrices of at most kGemvMaxElems weights, where its
// CTAs stream their 16 rows in one wave; above that the per-CTA fixed cost
// of several waves outweighs the split-K reduction it avoids.
constexpr long long kGemvMaxElems = 8ll << 20;
constexpr int kGemvThreads = 256;

__device__ __forceinline__ void fma8(float& acc, const uint4& w, const uint4& x) {
  const __nv_bfloat162* a = reinterpret_cast<const __nv_bfloat162*>(&w);
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 fa = __bfloat1622float2(a[i]), fb = __bfloat1622float2(b[i]);
    acc = fmaf(fa.x, fb.x, acc);
    acc = fmaf(fa.y, fb.y, acc);
  }
}

__global__ void __launch_bounds__(kGemvThreads, 2)
    k_gemv_bf16(const __nv_bfloat16* __restrict__ W, const __nv_bfloat16* __restrict__ X, int K, int nr, EpArgs ep,
           Ctrl* ctrl) {
  __shared__ __align__(16) float st[kGemvRows * kStP];   // [row][kStP] like the tensor-core partial tile
  __shared__ __align__(16) float par[4 * 64];
  __shared__ float red[4][2][32];
  cg::cluster_group cl = cg::this_cluster();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (ep.stall_ns) {
    // failure-detection test hook (see EpArgs::stall_ns): a bounded wait on a
    // barrier nothing arrives on runs out; nothing is in flight
    __shared__ uint64_t never;
    if (tid == 0) {
      ptx::mbar_init(&never, 1);
      ptx::fence_barrier_init();
      if (!ptx::mbar_wait(&never, 0, ep.stall_ns)) latch_error(ctrl, kErrTimeout, 104);
    }
    __syncthreads();
    ptx::grid_dep_wait();
    return;
  }
  const int tile = blockIdx.x >> 3, q = blockIdx.x & 7;
  const int n0 = tile * kBM, p0 = 8 * q;
  const int g = warp >> 1, kl = (warp & 1) * 32 + lane;  // row group, K lane
  // the group's 4 weight rows: features p0 + 4g' + i of the tile, where the
  // first two groups take features p0..p0+7 and the last two p0+64..p0+71
  const int fbase = (g < 2 ? p0 + 4 * g : 64 + p0 + 4 * (g - 2));
  const __nv_bfloat16* wr[4];
  bool wv[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    wv[i] = n0 + fbase + i < ep.n_out;
    wr[i] = W + (size_t)(wv[i] ? n0 + fbase + i : 0) * K;
  }
  const int nk8 = K >> 3;
  float acc[4][kGemvRows];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int m = 0; m < kGemvRows; ++m) acc[i][m] = 0.f;
  const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
  // weights of the first two chunks do not depend on the previous kernel
  uint4 w0[4], w1[4];
  int c = kl;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    w0[i] = (c < nk8 && wv[i]) ? __ldg(reinterpret_cast<const uint4*>(wr[i]) + c) : z4;
    w1[i] = (c + 64 < nk8 && wv[i]) ? __ldg(reinterpret_cast<const uint4*>(wr[i]) + c + 64) : z4;
  }
  if (tid < 64) stage_params(ep, par, n0, p0, 8, tid);
  ptx::grid_dep_wait();
  for (; c < nk8; c += 128) {
    // the next two chunks' weights are requested before this pair is used
    uint4 n0w[4], n1w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      n0w[i] = (c + 128 < nk8 && wv[i]) ? __ldg(reinterpret_cast<const uint4*>(wr[i]) + c + 128) : z4;
      n1w[i] = (c + 192 < nk8 && wv[i]) ? __ldg(reinterpret_cast<const uint4*>(wr[i]) + c + 192) : z4;
    }
    const bool c1 = c + 64 < nk8;
#pragma unroll
    for (int m = 0; m < kGemvRows; ++m) {
      if (m < nr) {
        const uint4* xr = reinterpret_cast<const uint4*>(X + (size_t)m * K);
        const uint4 x0 = xr[c], x1 = c1 ? xr[c + 64] : z4;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          fma8(acc[i][m], w0[i], x0);
          fma8(acc[i][m], w1[i], x1);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w0[i] = n0w[i];
      w1[i] = n1w[i];
    }
  }
  ptx::grid_dep_launch();
  // butterfly reduce-scatter over the warp: 32 values (4 rows x 8 stacked
  // rows, v = 8 i + m) leave lane l holding the warp's sum of value l
  float v[32];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int m = 0; m < kGemvRows; ++m) v[8 * i + m] = acc[i][m];
#pragma unroll
  for (int o = 16, len = 32; o >= 1; o >>= 1, len >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (j < len / 2) {
        const float send = upper ? v[j] : v[j + len / 2];
        const float keep = upper ? v[j + len / 2] : v[j];
        v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
  }
  red[g][warp & 1][lane] = v[0];
  __syncthreads();
  if (tid < 128) {
    const int gg = tid >> 5, vv = tid & 31, i = vv >> 3, m = vv & 7;
    const float sum = red[gg][0][vv] + red[gg][1][vv];
    const int f = (gg < 2 ? p0 + 4 * gg : 64 + p0 + 4 * (gg - 2)) + i;
    st[m * kStP + f] = sum;
  }
  __syncthreads();
  epilogue(ep, cl, st, par, 1, n0, p0, p0 + 8, tid, kGemvThreads, nullptr, 0);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D bf16 tensor map over a row-major [rows][cols] matrix with a box of
// 64 columns x box_rows rows and 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int tiles_of(int n_out) { return (n_out + kBM - 1) / kBM; }

// K-splits per tile (= cluster size).  `per_sm` CTAs fit on an SM (from the
// shared-memory footprint).  With two per SM, use them when each split still
// streams at least 16 K blocks (one CTA per SM cannot saturate HBM on a long
// K loop); otherwise aim at one wave of one CTA per SM with clusters of at
// most 8, since wider clusters cost more in launch, barrier and reduction
// than short K loops gain.
int choose_splits(int n_out, int K, int sms, int per_sm) {
  const int tiles = tiles_of(n_out), kb = K / kBK;
  int s = (per_sm >= 2 ? 2 * sms : sms) / tiles;
  if (s > kMaxSplit) s = kMaxSplit;
  if (per_sm >= 2 && s >= 1 && kb / s >= 16) return s;
  s = sms / tiles;
  if (s > 8) s = 8;
  if (s > kb / 2) s = kb / 2;
  if (s < 1) s = 1;
  return s;
}

// K-splits for a wide tile (more than 128 stacked rows): its footprint
// allows one CTA per SM, and a cluster must fit in one GPC, so a split count
// whose clusters the device cannot hold at once (max_clusters[s], measured
// for this kernel and footprint, less two clusters of headroom for the
// neighbouring kernels' CTAs that programmatic dependent launch keeps
// resident) would run in two waves.  The largest split count up to 8 that
// still gives each split at least eight K blocks and fits one wave is
// taken.  (Measured at 256 rows, six layers of dense24l_b128: QKV and Wo
// with K = 2048 took 13.4 / 12.9 us per launch at 5 / 6 splits and 12.5 /
// 12.2 us at 4, the step 1.556 -> 1.528 ms for Wo alone; down with K = 8192
// was fastest at 6 splits.)
int choose_splits_wide(int n_out, int K, int sms, const int* max_clusters) {
  const int tiles = tiles_of(n_out), kb = K / kBK;
  for (int s = 8; s > 1; --s) {
    if (kb / s < 8 || tiles * s > sms) continue;
    if (tiles <= max_clusters[s] - 2) return s;
  }
  return 1;
}

// Ring depth: as many stages as fit in `kb` KB (at least 2).
int stages_for(int N, int kb = 64) {
  int st = (kb * 1024) / (kStageW + N * kBK * 2);
  if (st > kMaxStages) st = kMaxStages;
  if (st < 2) st = 2;
  return st;
}

size_t smem_bytes(int N, int stages, bool direct = false) {
  size_t region = (size_t)stages * (kStageW + N * kBK * 2);
  if (!direct && (size_t)N * kStP * 4 > region) region = (size_t)N * kStP * 4;  // epilogue partial tile
  return region + 1024 + 4 * 64 * 4 + 256;
}

int mpad_of(const Dims& D) { return (2 * D.maxB + 15) / 16 * 16; }

}  // namespace

size_t tc_tickets_needed(const Dims&) { return 1; }

// Global split partials: one [N][kStP] tile per CTA of a split launch, at
// most two CTAs per SM (one for a wide tile), for every batch up to maxB.
size_t tc_partial_floats(const Dims& D) {
  if (!D.bf16 || D.hd != 128) return 0;
  const size_t mpad = (size_t)mpad_of(D);
  const size_t narrow = 2 * (mpad < (size_t)kWideN ? mpad : (size_t)kWideN);
  return (size_t)D.sms * (mpad > narrow ? mpad : narrow) * kStP;
}

bool tc_plan_init(TcPlan& P, const Dims& D, const Buffers& Bf, const std::vector<const void*>& wqkv,
                  const std::vector<const void*>& wo, const std::vector<const void*>& wgu,
                  const std::vector<const void*>& wd, const void* lm_head, std::string* err) {
  P.enabled = false;
  const char* e = getenv("DF_NO_TC");
  if (e && e[0] == '1') return true;
  const char* st = getenv("DF_TEST_GEMM_STALL_NS");
  P.stall_ns = st ? strtoull(st, nullptr, 10) : 0;
  const char* gr = getenv("DF_GEMV_ROWS");
  P.gemv_max_rows = gr ? atoi(gr) : 2;
  if (!D.bf16) return true;
  if (D.hd != 128) return true;
  if (D.qdim % kBM || D.kvdim % kBM || D.d % kBM || D.d % kBK || D.qdim % kBK) return true;
  if (!D.E && (D.F % kBK)) return true;
  if (mpad_of(D) > 256) return true;
  if (!encode_fn()) return true;
  const int Mpad = mpad_of(D);
  P.w_qkv.resize(D.L);
  P.w_o.resize(D.L);
  bool ok = true;
  for (int l = 0; l < D.L; ++l) {
    ok &= make_map(&P.w_qkv[l], wqkv[l], D.d, D.qkvn, kBM);
    ok &= make_map(&P.w_o[l], wo[l], D.qdim, D.d, kBM);
  }
  if (!D.E) {
    P.w_gu.resize(D.L);
    P.w_d.resize(D.L);
    for (int l = 0; l < D.L; ++l) {
      ok &= make_map(&P.w_gu[l], wgu[l], D.d, 2 * D.F, kBM);
      ok &= make_map(&P.w_d[l], wd[l], D.F, D.d, kBM);
    }
  }
  ok &= make_map(&P.w_lm, lm_head, D.d, D.V, kBM);
  if (!ok) {
    if (err) *err = "cuTensorMapEncodeTiled failed for a weight matrix";
    return false;
  }
  P.u_ptr = Bf.u;
  P.o_ptr = Bf.o;
  P.z_ptr = Bf.z;
  P.mpad = Mpad;
  cudaFuncSetAttribute(k_tc_gemm<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  cudaFuncSetAttribute(k_tc_gemm<128>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  cudaFuncSetAttribute(k_tc_gemm<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  cudaFuncSetAttribute(k_tc_gemm<256>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  cudaFuncSetAttribute(k_tc_gemm<512>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  cudaFuncSetAttribute(k_tc_gemm<512>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  cudaFuncSetAttribute(k_tc_gemm<128, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  P.enabled = true;
  P.dense = !D.E;
  return true;
}

bool tc_plan_batch(TcPlan& P, const Dims& D, int B, std::string* err) {
  P.B = B;
  if (!P.enabled) return true;
  // Few stacked rows: the CUDA-core GEMV for the matrices where it measured
  // faster than the tensor-core tile (see gemv_max_rows)
  const bool few = 2 * B <= P.gemv_max_rows && 2 * B <= kGemvRows;
  auto small = [&](long long n_out, long long K) { return n_out * K <= kGemvMaxElems; };
  P.gemv[(int)TcOp::QKV] = few && small(D.qkvn, D.d);
  P.gemv[(int)TcOp::RESID] = few && small(D.d, D.qdim);
  P.gemv[(int)TcOp::SWIGLU] = few && !D.E && small(2LL * D.F, D.d);
  P.gemv[(int)TcOp::DOWN] = few && !D.E && small(D.d, D.F);
  P.gemv[(int)TcOp::LOGITS] = few && small(D.V, D.d);
  int N = (2 * B + 15) / 16 * 16;
  P.npad = N;
  // the split plan depends on how many CTAs of this N fit on one SM
  P.sms = D.sms;
  if (N > kWideN) {
    // clusters of each size the device holds at once at the wide footprint
    int maxc[9] = {0};
    const size_t smem = smem_bytes(N, stages_for(N, kWideKB));
    for (int sz = 1; sz <= 8; ++sz) {
      cudaLaunchConfig_t lc{};
      lc.gridDim = dim3(sz);
      lc.blockDim = dim3(512);
      lc.dynamicSmemBytes = smem;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = sz;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      lc.attrs = at;
      lc.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, k_tc_gemm<512>, &lc) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
      }
      maxc[sz] = n;
    }
    P.splits[(int)TcOp::QKV] = choose_splits_wide(D.qkvn, D.d, D.sms, maxc);
    P.splits[(int)TcOp::RESID] = choose_splits_wide(D.d, D.qdim, D.sms, maxc);
    P.splits[(int)TcOp::SWIGLU] = D.E ? 1 : choose_splits_wide(2 * D.F, D.d, D.sms, maxc);
    P.splits[(int)TcOp::DOWN] = D.E ? 1 : choose_splits_wide(D.d, D.F, D.sms, maxc);
    P.splits[(int)TcOp::LOGITS] = choose_splits_wide(D.V, D.d, D.sms, maxc);
  } else {
    const int per_sm = (int)((227 * 1024) / (smem_bytes(N, stages_for(N)) + 1024));
    P.splits[(int)TcOp::QKV] = choose_splits(D.qkvn, D.d, D.sms, per_sm);
    P.splits[(int)TcOp::RESID] = choose_splits(D.d, D.qdim, D.sms, per_sm);
    P.splits[(int)TcOp::SWIGLU] = D.E ? 1 : choose_splits(2 * D.F, D.d, D.sms, per_sm);
    P.splits[(int)TcOp::DOWN] = D.E ? 1 : choose_splits(D.d, D.F, D.sms, per_sm);
    P.splits[(int)TcOp::LOGITS] = choose_splits(D.V, D.d, D.sms, per_sm);
  }
  bool ok = make_map(&P.x_u, P.u_ptr, D.d, P.mpad, N) && make_map(&P.x_o, P.o_ptr, D.qdim, P.mpad, N);
  if (P.dense) ok = ok && make_map(&P.x_z, P.z_ptr, D.F, P.mpad, N);
  if (!ok && err) *err = "cuTensorMapEncodeTiled failed for an activation buffer";
  return ok;
}

void tc_plan_free(TcPlan& P) {
  P.w_qkv.clear();
  P.w_o.clear();
  P.w_gu.clear();
  P.w_d.clear();
}

bool tc_can_run(const TcPlan& P, TcOp op) {
  if (!P.enabled) return false;
  if ((op == TcOp::SWIGLU || op == TcOp::DOWN) && !P.dense) return false;
  return true;
}

namespace {

EpArgs base_args(const Dims& D, const Buffers& Bf, const Rows& R, TcOp op, int n_out) {
  EpArgs ep{};
  ep.op = (int)op;
  ep.lo = R.lo;
  ep.hi = R.hi;
  ep.B = R.B;
  ep.n_out = n_out;
  ep.rope = Bf.rope;
  ep.ctrl = Bf.ctrl;
  ep.qatt = Bf.qatt;
  ep.qdim = D.qdim;
  ep.kvdim = D.kvdim;
  ep.hd = D.hd;
  ep.Hkv = D.Hkv;
  ep.km = Bf.kvm;
  ep.h = Bf.h;
  ep.d = D.d;
  ep.z = (__nv_bfloat16*)Bf.z;
  ep.F = D.F;
  ep.logits = Bf.logits;
  ep.V = D.V;
  ep.gpart = Bf.gpart;
  return ep;
}

void launch(const TcPlan& P, const CUtensorMap& tw, const CUtensorMap& tx, const void* w, const void* x, int n_out,
            int K, const EpArgs& ep0, const Buffers& Bf, cudaStream_t s, int splits) {
  EpArgs ep = ep0;
  ep.stall_ns = P.stall_ns;
  if (P.gemv[ep.op]) {
    // a few stacked rows: CUDA-core GEMV, 8 feature pairs per CTA, no split
    launch_pdl(k_gemv_bf16, dim3(tiles_of(n_out) * 8), dim3(kGemvThreads), 0, s,
               static_cast<const __nv_bfloat16*>(w), static_cast<const __nv_bfloat16*>(x), K, 2 * P.B, ep, Bf.ctrl);
    return;
  }
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(tiles_of(n_out) * splits);
  lc.blockDim = dim3(128);
  // ~64 KB rings let two GEMM CTAs and a neighbouring kernel's CTA share an
  // SM; a launch of at most one CTA per SM may use a deeper ring, and a wide
  // tile (its partial tile alone takes half the SM) the deepest.  The LM
  // head of a wide batch has more tiles than SMs and no K-split: its logits
  // leave straight from TMEM, and a two-stage ring lets two CTAs share an SM
  // so that the launch runs in one wave instead of two.
  const bool direct = ep.op == (int)TcOp::LOGITS && splits == 1 && P.npad > kWideN && tiles_of(n_out) > P.sms;
  const bool one_per_sm = tiles_of(n_out) * splits <= P.sms;
  const int stages =
      direct ? 2 : stages_for(P.npad, P.npad > kWideN ? kWideKB : one_per_sm ? DF_GEMM_WIDE_KB : 64);
  lc.dynamicSmemBytes = smem_bytes(P.npad, stages, direct);
  lc.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = splits;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  lc.attrs = at;
  lc.numAttrs = 2;
  // a footprint above half the SM already means one CTA per SM: use the
  // wider CTA, whose extra warps share the epilogue
  if (direct) {
    // LOGITS straight from TMEM (k_tc_gemm<128, true>): no partial tile
    cudaLaunchKernelEx(&lc, k_tc_gemm<128, true>, tw, tx, P.npad, K / kBK, stages, ep, Bf.ctrl);
  } else if (P.npad > kWideN) {
    // 256 stacked rows: 16 warps share the TMEM drain and the epilogue
    lc.blockDim = dim3(512);
    cudaLaunchKernelEx(&lc, k_tc_gemm<512>, tw, tx, P.npad, K / kBK, stages, ep, Bf.ctrl);
  } else if (lc.dynamicSmemBytes > 114 * 1024) {
    lc.blockDim = dim3(256);
    cudaLaunchKernelEx(&lc, k_tc_gemm<256>, tw, tx, P.npad, K / kBK, stages, ep, Bf.ctrl);
  } else {
    cudaLaunchKernelEx(&lc, k_tc_gemm<128>, tw, tx, P.npad, K / kBK, stages, ep, Bf.ctrl);
  }
}

}  // namespace

void tc_qkv(const TcPlan& P, const Dims& D, const Buffers& Bf, const void* w, const float* a, void* kv, int layer,
            const Couple& C, const Rows& R, cudaStream_t s) {
  (void)w;
  EpArgs ep = base_args(D, Bf, R, TcOp::QKV, D.qkvn);
  ep.a = a;
  ep.C = C;
  ep.kv = (__nv_bfloat16*)kv;
  ep.layer = layer;
  launch(P, P.w_qkv[layer], P.x_u, w, P.u_ptr, D.qkvn, D.d, ep, Bf, s, P.splits[(int)TcOp::QKV]);
}

void tc_resid(const TcPlan& P, const Dims& D, const Buffers& Bf, const void* w, int layer, const Rows& R,
              cudaStream_t s) {
  (void)w;
  EpArgs ep = base_args(D, Bf, R, TcOp::RESID, D.d);
  launch(P, P.w_o[layer], P.x_o, w, P.o_ptr, D.d, D.qdim, ep, Bf, s, P.splits[(int)TcOp::RESID]);
}

void tc_swiglu(const TcPlan& P, const Dims& D, const Buffers& Bf, const void* w, int layer, const float* bvec,
               const Couple& C, const Rows& R, cudaStream_t s) {
  (void)w;
  EpArgs ep = base_args(D, Bf, R, TcOp::SWIGLU, 2 * D.F);
  ep.bvec = bvec;
  ep.C = C;
  launch(P, P.w_gu[layer], P.x_u, w, P.u_ptr, 2 * D.F, D.d, ep, Bf, s, P.splits[(int)TcOp::SWIGLU]);
}

void tc_down(const TcPlan& P, const Dims& D, const Buffers& Bf, const void* w, int layer, const float* cvec,
             const Couple& C, const Rows& R, cudaStream_t s) {
  (void)w;
  EpArgs ep = base_args(D, Bf, R, TcOp::DOWN, D.d);
  ep.cvec = cvec;
  ep.C = C;
  launch(P, P.w_d[layer], P.x_z, w, P.z_ptr, D.d, D.F, ep, Bf, s, P.splits[(int)TcOp::DOWN]);
}

void tc_logits(const TcPlan& P, const Dims& D, const Buffers& Bf, const void* w, const Rows& R, cudaStream_t s) {
  (void)w;
  EpArgs ep = base_args(D, Bf, R, TcOp::LOGITS, D.V);
  launch(P, P.w_lm, P.x_u, w, P.u_ptr, D.V, D.d, ep, Bf, s, P.splits[(int)TcOp::LOGITS]);
}

}  // namespace df
