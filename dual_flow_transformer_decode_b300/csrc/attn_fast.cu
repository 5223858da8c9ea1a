// Split-KV shared-KV decode attention for bf16 caches with head_dim 128.
//
// "Mecanismos Clave" (Atención de KV Compartido Asimétrico): the auxiliary
// query Q2 attends to the primary K1/V1, so one pass over a KV head's cache
// serves the G primary and G auxiliary query heads of that KV head.
//
// Grid (split, kv head, sequence); the splits of one (sequence, KV head)
// form a thread-block cluster.  A producer warp streams 64-position K and V
// tiles with TMA (3-D tensor map over the cache, 128-byte swizzle) through a
// 2-stage mbarrier ring (up to 4); tiles below the current position t do not depend on
// the previous kernel and are requested before griddepcontrol.wait.  Each
// tile is read from HBM once for all query rows of the KV head (up to 16:
// G primary + G auxiliary).  Four compute warps each own 16 positions of a
// tile and run on the tensor cores (mma.sync m16n8k16, fp32 accumulate):
//   S = Q · K^T    Q is bf16 by construction (the oracle rounds it too), so
//                  the products are exact;
//   online softmax per row in fp32;
//   O += P · V     P is split into bf16 hi + lo parts and both are applied,
//                  so P enters with ~16 significant bits (relative error below
//                  2^-16) — far below the bf16 rounding of o that follows.
//                  With at most 8 query rows (2G <= 8) the lo parts ride in
//                  the m16 tile's idle rows 8..15, so one MMA applies both
//                  parts, and the two halves are added after the last tile.
// The warps' (m, l, O) are merged in shared memory; the splits are merged
// through distributed shared memory in split order (rank r merges a slice of
// the output) and written as bf16 rows of o.  Each query row's result
// depends only on that row, so the primary rows do not change with the set
// of active auxiliary rows.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cooperative_groups.h>
#include <math.h>

#include <cmath>
#include <stdlib.h>

#include "attn_fast.h"
#include "ptx.cuh"

namespace df {

namespace cg = cooperative_groups;

namespace {

constexpr int HD = 128;
constexpr int TP = 64;            // positions per tile
constexpr int NSMAX = 4;          // ring stages (runtime NS <= NSMAX)
constexpr int BOX = TP * 64 * 2;  // one TMA box: 64 positions x 64 dims bf16 = 8 KB
constexpr int STAGE = 4 * BOX;    // K lo, K hi, V lo, V hi = 32 KB
constexpr int RQ = 16;            // query rows per MMA (m16)
constexpr int kMaxSplits = 16;    // cluster size limit
constexpr int kShortStages = 2;   // ring stages when a split has few tiles
constexpr int kLongStages = 3;    // ... and when it has at least kLongTiles
constexpr int kLongTiles = 8;
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

__device__ __forceinline__ uint32_t pack_bf16(float lo_elem, float hi_elem) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo_elem, hi_elem);
  return *reinterpret_cast<uint32_t*>(&v);
}

// p = hi + lo with hi = bf16(p), lo = bf16(p - hi), packed in pairs.
__device__ __forceinline__ void split_pair(float x, float y, uint32_t& hi, uint32_t& lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  float2 hf = __bfloat1622float2(h);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = pack_bf16(x - hf.x, y - hf.y);
}

// Byte offset of (position, dim) inside a K or V tile made of two 128-byte
// swizzled boxes (dims 0..63, 64..127).
__device__ __forceinline__ uint32_t sw_off(int pos, int dim) {
  int box = dim >> 6, dd = dim & 63;
  return box * BOX + pos * 128 + ((((dd >> 3) ^ (pos & 7)) << 4)) + ((dd & 7) << 1);
}

__global__ void __launch_bounds__(160, 2)
    k_attn_tma(const __grid_constant__ CUtensorMap tkv, const float* __restrict__ qatt, Ctrl* __restrict__ ctrl,
               __nv_bfloat16* __restrict__ out, int B, int Hkv, int G, KvMap km, int layer, int flo, int fhi,
               int NS, int l2pf, int fold) {
  extern __shared__ uint8_t smem_raw[];
  cg::cluster_group cl = cg::this_cluster();
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = base;                                                    // NS * 32 KB
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(ring + NS * STAGE);  // [16][128]
  float* cpart = reinterpret_cast<float*>(qs + RQ * HD);                   // CTA partial: M[16], L[16], O[16][128]
  uint64_t* full = reinterpret_cast<uint64_t*>(cpart + 2 * RQ + RQ * HD);
  uint64_t* empty = full + NSMAX;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + NSMAX);

  const int splits = (int)cl.num_blocks();
  const int s = (int)cl.block_rank(), g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = (fhi - flo) * G;
  const int qdim = Hkv * G * HD;

  // Positions 0..t of this sequence: the cache below t was written by earlier
  // steps, position t by the QKV kernel this kernel depends on.
  const int t = kv_seq_pos(km, ctrl, b);
  const int n = t + 1;
  int chunk = (n + splits - 1) / splits;
  chunk = (chunk + TP - 1) / TP * TP;
  const int s0 = s * chunk, s1 = min(n, s0 + chunk);
  const int ntiles = s1 > s0 ? (s1 - s0 + TP - 1) / TP : 0;
  // tensor-map rows (z) of the K and V blocks of the page holding position
  // p0, and the position's offset in it (y); a 64-position tile never spans
  // two pages (pages hold a multiple of 64 positions)
  auto tile_z = [&](int p0, int kvsel) { return ((layer * 2 + kvsel) * km.NP + kv_page(km, b, p0)) * Hkv + g; };

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&empty[i], 4);
    }
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
  }
  __syncthreads();

  // Producer, part 1: the first tiles, if they lie below position t.
  int issued = 0;
  if (warp == 4 && lane == 0) {
    ptx::prefetch_tmap(&tkv);
    const int pre = ntiles < NS ? ntiles : NS;
    for (; issued < pre; ++issued) {
      const int p0 = s0 + issued * TP;
      if (p0 + TP > t) break;
      const int zK = tile_z(p0, 0), zV = tile_z(p0, 1), y = kv_off(km, p0);
      uint8_t* dst = ring + issued * STAGE;
      ptx::mbar_arrive_expect_tx(&full[issued], STAGE);
      ptx::tma_load_3d(dst + 0 * BOX, &tkv, &full[issued], 0, y, zK);
      ptx::tma_load_3d(dst + 1 * BOX, &tkv, &full[issued], 64, y, zK);
      ptx::tma_load_3d(dst + 2 * BOX, &tkv, &full[issued], 0, y, zV);
      ptx::tma_load_3d(dst + 3 * BOX, &tkv, &full[issued], 64, y, zV);
    }
    if (l2pf)
      for (int i = issued; i < ntiles; ++i) {
        const int p0 = s0 + i * TP;
        if (p0 + TP > t) break;
        const int zK = tile_z(p0, 0), zV = tile_z(p0, 1), y = kv_off(km, p0);
        ptx::tma_prefetch_3d(&tkv, 0, y, zK);
        ptx::tma_prefetch_3d(&tkv, 64, y, zK);
        ptx::tma_prefetch_3d(&tkv, 0, y, zV);
        ptx::tma_prefetch_3d(&tkv, 64, y, zV);
      }
  }
  ptx::grid_dep_wait();

  // Query rows (bf16 values) -> shared memory [16][128]; rows >= R are zero.
  {
    float4 qv[(RQ * HD / 4) / 160 + 1];
#pragma unroll
    for (int k = 0; k < (RQ * HD / 4) / 160 + 1; ++k) {
      const int idx = tid + k * 160;
      qv[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (idx < RQ * HD / 4) {
        const int r = idx / (HD / 4), i4 = idx % (HD / 4);
        if (r < R) {
          const int f = flo + r / G, j = r % G;
          qv[k] = *reinterpret_cast<const float4*>(qatt + (size_t)(f * B + b) * qdim + (g * G + j) * HD + 4 * i4);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < (RQ * HD / 4) / 160 + 1; ++k) {
      const int idx = tid + k * 160;
      if (idx < RQ * HD / 4) {
        __nv_bfloat162* d = reinterpret_cast<__nv_bfloat162*>(qs + 4 * idx);
        d[0] = __floats2bfloat162_rn(qv[k].x, qv[k].y);
        d[1] = __floats2bfloat162_rn(qv[k].z, qv[k].w);
      }
    }
  }
  __syncthreads();

  if (warp == 4) {
    // Producer, part 2: the remaining tiles through the ring.
    if (lane == 0) {
      for (int i = issued; i < ntiles; ++i) {
        const int st = i % NS;
        if (i >= NS && !ptx::mbar_wait(&empty[st], ((i / NS) - 1) & 1)) {
          *abort_flag = 1;
          latch_error(ctrl, kErrTimeout, 200);
          break;
        }
        if (*abort_flag) break;
        const int p0 = s0 + i * TP;
        const int zK = tile_z(p0, 0), zV = tile_z(p0, 1), y = kv_off(km, p0);
        uint8_t* dst = ring + st * STAGE;
        ptx::mbar_arrive_expect_tx(&full[st], STAGE);
        ptx::tma_load_3d(dst + 0 * BOX, &tkv, &full[st], 0, y, zK);
        ptx::tma_load_3d(dst + 1 * BOX, &tkv, &full[st], 64, y, zK);
        ptx::tma_load_3d(dst + 2 * BOX, &tkv, &full[st], 0, y, zV);
        ptx::tma_load_3d(dst + 3 * BOX, &tkv, &full[st], 64, y, zV);
        issued = i + 1;
      }
      if (*abort_flag) {
        // let copies still in flight land before the shared memory is released
        for (int i = issued - NS < 0 ? 0 : issued - NS; i < issued; ++i)
          ptx::mbar_wait(&full[i % NS], (i / NS) & 1, 100000000ull);
      }
    }
    __syncwarp();
  }

  const int gq = lane >> 2, tq = lane & 3;  // mma fragment coordinates
  float m_run[2] = {-INFINITY, -INFINITY};  // rows gq, gq+8
  float l_run[2] = {0.f, 0.f};
  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

  if (warp < 4) {
    // Q as the A operand: rows gq, gq+8; dims kk*16 + 2tq (+8)
    uint32_t qa[8][4];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const __nv_bfloat16* q0 = qs + gq * HD + kk * 16 + 2 * tq;
      const __nv_bfloat16* q1 = qs + (gq + 8) * HD + kk * 16 + 2 * tq;
      qa[kk][0] = *reinterpret_cast<const uint32_t*>(q0);
      qa[kk][1] = *reinterpret_cast<const uint32_t*>(q1);
      qa[kk][2] = *reinterpret_cast<const uint32_t*>(q0 + 8);
      qa[kk][3] = *reinterpret_cast<const uint32_t*>(q1 + 8);
    }
    const int mq = lane >> 3, r8 = lane & 7;  // ldmatrix: matrix index, row in matrix
    for (int it = 0; it < ntiles; ++it) {
      const int st = it % NS;
      if (!ptx::mbar_wait(&full[st], (it / NS) & 1)) {
        *abort_flag = 1;
        latch_error(ctrl, kErrTimeout, 201);
        break;
      }
      if (*abort_flag) break;
      const uint32_t kbase = ptx::smem_u32(ring + st * STAGE);
      const uint32_t vbase = kbase + 2 * BOX;
      // ---- S[16 rows][16 positions] for positions 16*warp .. +15; dims
      // 0..63 and 64..127 accumulate separately (four independent MMA
      // chains instead of two), then add
      float sc[2][4], sd[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
        sd[nt][0] = sd[nt][1] = sd[nt][2] = sd[nt][3] = 0.f;
      }
      const int kpos = warp * 16 + (mq >> 1) * 8 + r8;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t b00, b01, b10, b11;  // n-tile 0: (b0, b1), n-tile 1: (b0, b1)
        uint32_t c00, c01, c10, c11;
        ldsm_x4(kbase + sw_off(kpos, kk * 16 + (mq & 1) * 8), b00, b01, b10, b11);
        ldsm_x4(kbase + sw_off(kpos, (kk + 4) * 16 + (mq & 1) * 8), c00, c01, c10, c11);
        mma_16816(sc[0], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b00, b01);
        mma_16816(sc[1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b10, b11);
        mma_16816(sd[0], qa[kk + 4][0], qa[kk + 4][1], qa[kk + 4][2], qa[kk + 4][3], c00, c01);
        mma_16816(sd[1], qa[kk + 4][0], qa[kk + 4][1], qa[kk + 4][2], qa[kk + 4][3], c10, c11);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[nt][e] += sd[nt][e];
      // ---- online softmax for rows gq (c0, c1) and gq+8 (c2, c3); with
      // fold, rows gq + 8 hold no query and are skipped
      const int pbase = s0 + it * TP + warp * 16 + 2 * tq;
      float corr[2] = {1.f, 1.f};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (fold && h == 1) break;
        float v[4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int pos = pbase + nt * 8 + e;
            v[nt * 2 + e] = pos < s1 ? sc[nt][2 * h + e] * kScale : -INFINITY;
          }
        float mx = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mo = m_run[h], mn = fmaxf(mo, mx);
        // the fast exponential (ex2-based, a few ulp): P enters P·V with
        // 16 significant bits anyway
        corr[h] = (mo == -INFINITY) ? 0.f : __expf(mo - mn);
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          v[k] = (v[k] == -INFINITY) ? 0.f : __expf(v[k] - mn);
          sum += v[k];
        }
        m_run[h] = mn;
        l_run[h] = l_run[h] * corr[h] + sum;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          sc[nt][2 * h] = v[nt * 2];
          sc[nt][2 * h + 1] = v[nt * 2 + 1];
        }
      }
      // ---- P as the A operand (16 rows x 16 positions), hi and lo parts
      uint32_t ph[4], pl[4];
      split_pair(sc[0][0], sc[0][1], ph[0], pl[0]);  // row gq,   positions 2tq..
      split_pair(sc[0][2], sc[0][3], ph[1], pl[1]);  // row gq+8
      split_pair(sc[1][0], sc[1][1], ph[2], pl[2]);  // row gq,   positions 8+2tq..
      split_pair(sc[1][2], sc[1][3], ph[3], pl[3]);  // row gq+8
      const int vpos = warp * 16 + (mq & 1) * 8 + r8;
      if (fold) {
        // At most 8 query rows: the lo part of row gq takes the MMA's
        // otherwise idle row gq + 8, so one MMA applies both parts (rows
        // gq + 8 accumulate lo * V; they are added to rows gq at the end).
        // Once the running maxima settle every factor is 1 and the rescale
        // (exact either way) is skipped.
        if (__any_sync(0xffffffffu, corr[0] != 1.f)) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            o[j][0] *= corr[0];
            o[j][1] *= corr[0];
            o[j][2] *= corr[0];
            o[j][3] *= corr[0];
          }
        }
        // ---- O += P V: V^T fragments by ldmatrix.trans, two 8-dim n-tiles per load
#pragma unroll
        for (int j2 = 0; j2 < 8; ++j2) {
          uint32_t v00, v01, v10, v11;
          ldsm_x4_t(vbase + sw_off(vpos, j2 * 16 + (mq >> 1) * 8), v00, v01, v10, v11);
          mma_16816(o[2 * j2], ph[0], pl[0], ph[2], pl[2], v00, v01);
          mma_16816(o[2 * j2 + 1], ph[0], pl[0], ph[2], pl[2], v10, v11);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          o[j][0] *= corr[0];
          o[j][1] *= corr[0];
          o[j][2] *= corr[1];
          o[j][3] *= corr[1];
        }
#pragma unroll
        for (int j2 = 0; j2 < 8; ++j2) {
          uint32_t v00, v01, v10, v11;
          ldsm_x4_t(vbase + sw_off(vpos, j2 * 16 + (mq >> 1) * 8), v00, v01, v10, v11);
          mma_16816(o[2 * j2], ph[0], ph[1], ph[2], ph[3], v00, v01);
          mma_16816(o[2 * j2], pl[0], pl[1], pl[2], pl[3], v00, v01);
          mma_16816(o[2 * j2 + 1], ph[0], ph[1], ph[2], ph[3], v10, v11);
          mma_16816(o[2 * j2 + 1], pl[0], pl[1], pl[2], pl[3], v10, v11);
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty[st]);
    }
    if (fold) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        o[j][0] += o[j][2];
        o[j][1] += o[j][3];
        o[j][2] = o[j][3] = 0.f;
      }
    }
    // row sums over the four lanes of a row
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
    }
  }
  __syncthreads();
  ptx::grid_dep_launch();

  // ---- merge the four warps (reuse the ring): mw, lw, ew [4][16] and the
  // valid rows of ow [4][16][OWS] (row stride padded against bank conflicts)
  constexpr int OWS = HD + 8;
  float* mw = reinterpret_cast<float*>(ring);
  float* lw = mw + 4 * RQ;
  float* ew = lw + 4 * RQ;
  float* ow = ew + 4 * RQ;
  if (warp < 4) {
    if (tq == 0) {
      mw[warp * RQ + gq] = m_run[0];
      mw[warp * RQ + gq + 8] = m_run[1];
      lw[warp * RQ + gq] = l_run[0];
      lw[warp * RQ + gq + 8] = l_run[1];
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int dcol = j * 8 + 2 * tq;
      if (gq < R)
        *reinterpret_cast<float2*>(ow + ((size_t)warp * RQ + gq) * OWS + dcol) = make_float2(o[j][0], o[j][1]);
      if (gq + 8 < R)
        *reinterpret_cast<float2*>(ow + ((size_t)warp * RQ + gq + 8) * OWS + dcol) = make_float2(o[j][2], o[j][3]);
    }
  }
  __syncthreads();
  const bool aborted = *abort_flag != 0;
  // per row: the CTA maximum, each warp's weight relative to it, the sum
  if (tid < R) {
    const int r = tid;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, mw[w * RQ + r]);
    float l = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float mv = mw[w * RQ + r];
      const float e = (mv == -INFINITY) ? 0.f : expf(mv - M);
      ew[w * RQ + r] = e;
      l = fmaf(e, lw[w * RQ + r], l);
    }
    cpart[r] = M;
    cpart[RQ + r] = l;
  }
  __syncthreads();
  // CTA partial in cpart: M[16], L[16], O[16][128] (unnormalised)
  for (int idx = tid; idx < R * HD; idx += blockDim.x) {
    const int r = idx / HD, i = idx % HD;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) acc = fmaf(ew[w * RQ + r], ow[((size_t)w * RQ + r) * OWS + i], acc);
    cpart[2 * RQ + r * HD + i] = acc;
  }
  // ---- merge the splits of the cluster, in split order; rank s writes the
  // output elements [s*R*HD/splits, (s+1)*R*HD/splits).  Per row the splits'
  // weights and the denominator are formed once (sew, sden), then each
  // element reads only the splits' partial outputs.
  cl.sync();
  float* sew = reinterpret_cast<float*>(ring);  // [kMaxSplits][16]
  float* sden = sew + kMaxSplits * RQ;          // [16]
  const int tot = R * HD, e0 = s * tot / splits, e1 = (s + 1) * tot / splits;
  const int r0 = e0 / HD, r1 = e1 > e0 ? (e1 - 1) / HD + 1 : r0;
  if (!aborted && tid < r1 - r0) {
    const int r = r0 + tid;
    float ms[kMaxSplits], ls[kMaxSplits];
#pragma unroll
    for (int sp = 0; sp < kMaxSplits; ++sp)
      if (sp < splits) {
        const float* rp = cl.map_shared_rank(cpart, sp);
        ms[sp] = rp[r];
        ls[sp] = rp[RQ + r];
      }
    float M = -INFINITY;
#pragma unroll
    for (int sp = 0; sp < kMaxSplits; ++sp)
      if (sp < splits) M = fmaxf(M, ms[sp]);
    float den = 0.f;
#pragma unroll
    for (int sp = 0; sp < kMaxSplits; ++sp)
      if (sp < splits) {
        const float e = ms[sp] != -INFINITY ? expf(ms[sp] - M) : 0.f;
        sew[sp * RQ + r] = e;
        den = fmaf(e, ls[sp], den);
      }
    sden[r] = den;
  }
  __syncthreads();
  if (!aborted) {
    for (int idx = e0 + tid; idx < e1; idx += blockDim.x) {
      const int r = idx / HD, i = idx % HD;
      float os[kMaxSplits];
#pragma unroll
      for (int sp = 0; sp < kMaxSplits; ++sp)
        if (sp < splits) os[sp] = cl.map_shared_rank(cpart, sp)[2 * RQ + r * HD + i];
      float acc = 0.f;
#pragma unroll
      for (int sp = 0; sp < kMaxSplits; ++sp)
        if (sp < splits) acc = fmaf(sew[sp * RQ + r], os[sp], acc);
      const int f = flo + r / G, j = r % G;
      out[(size_t)(f * B + b) * qdim + (g * G + j) * HD + i] = __float2bfloat16_rn(acc / sden[r]);
    }
  }
  // keep this CTA's partial alive until the whole cluster has read it
  cl.sync();
}

size_t smem_bytes(int NS) {
  size_t ring = (size_t)NS * STAGE;
  size_t merge = (size_t)(3 * 4 * RQ + 4 * RQ * (HD + 8)) * 4;  // reuses the ring after the loop
  if (merge > ring) ring = merge;
  return 1024 + ring + (size_t)RQ * HD * 2 + (size_t)(2 * RQ + RQ * HD) * 4 + 2 * NSMAX * 8 + 16;
}

}  // namespace

bool attn_fast_init(AttnPlan& P, const Dims& D, void* kv, std::string* err) {
  P.enabled = false;
  const char* e = getenv("DF_NO_FAST_ATTN");
  if (e && e[0] == '1') return true;
  if (!D.bf16 || D.hd != HD || 2 * D.G > RQ) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return true;
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  // (head_dim, positions of a page, L * 2 * pages * KV heads)
  cuuint64_t dims[3] = {(cuuint64_t)HD, (cuuint64_t)D.PG, (cuuint64_t)D.L * 2 * D.NP * D.Hkv};
  cuuint64_t strides[2] = {(cuuint64_t)HD * 2, (cuuint64_t)D.PG * HD * 2};
  cuuint32_t box[3] = {64, TP, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(&P.kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kv, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (err) *err = "cuTensorMapEncodeTiled failed for the KV cache";
    return false;
  }
  cudaFuncSetAttribute(k_attn_tma, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes(NSMAX));
  cudaFuncSetAttribute(k_attn_tma, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  // How many clusters of each size fit on the device at once.  A cluster's
  // CTAs must share one GPC, so large clusters fit fewer times than the
  // per-SM occupancy alone suggests.
  for (int sp = 1; sp <= kMaxSplits; ++sp) {
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(sp, 1, 1);
    lc.blockDim = dim3(160);
    lc.dynamicSmemBytes = smem_bytes(kShortStages);  // split launches use the short ring
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = sp;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    lc.attrs = at;
    lc.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (void*)k_attn_tma, &lc) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    P.max_clusters[sp] = n;
  }
  P.enabled = true;
  return true;
}

int attn_fast_splits(const AttnPlan& P, const Dims& D, int B) {
  const int pairs = B * D.Hkv;
  const int T = (D.max_len + 63) / 64;
  const double c0 = 4.0, c_tile = 1.5;  // as in attn_splits
  int best = 1;
  double best_t = 1e30;
  for (int sp = 1; sp <= kMaxSplits && sp <= T; ++sp) {
    // two clusters of headroom: the CTAs of the neighbouring kernels that
    // programmatic dependent launch keeps resident displace some (measured at
    // 16 pairs: 13-CTA clusters, 17 held on an idle device, ran 8% slower
    // than 12-CTA clusters, 21 held)
    const int cap = (P.max_clusters[sp] > 0 ? P.max_clusters[sp] : (2 * D.sms) / sp) - 2;
    if (cap <= 0) break;
    const double waves = std::ceil((double)pairs / cap);
    const double tm = waves * (c0 + std::ceil((double)T / sp) * c_tile);
    if (tm < best_t - 1e-9) {
      best_t = tm;
      best = sp;
    }
  }
  return best;
}

void attn_fast_free(AttnPlan& P) { P.enabled = false; }

bool attn_fast_can_run(const AttnPlan& P, const Dims& D) { return P.enabled && D.hd == HD && 2 * D.G <= RQ; }

int attn_fast_max_splits() { return kMaxSplits; }

void attn_fast(const AttnPlan& P, const Dims& D, const Buffers& Bf, const void* kv, int layer, int splits,
               const Rows& R, cudaStream_t s) {
  (void)kv;
  const int flo = R.lo >= R.B ? 1 : 0, fhi = R.hi > R.B ? 2 : 1;
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(splits, D.Hkv, R.B);
  lc.blockDim = dim3(160);
  // Ring depth: three 32 KB stages for an unsplit launch whose CTAs stream
  // at least kLongTiles tiles (over the context capacity, so one captured
  // launch serves every position), else two.  Measured inside the whole
  // step: batch 128 at 4096 positions 6.040 -> 6.014 ms per step with three;
  // at 32768 positions in 12-CTA clusters three stages were 47 against 53 us
  // per launch alone but 2.045 against 1.604 ms per step, because the larger
  // clusters then wait for the neighbouring kernels' resident CTAs to leave.
  // L2 prefetch of the split measured no faster.
  const int tiles_per_split = ((D.max_len + TP - 1) / TP + splits - 1) / splits;
  const int ns = (splits == 1 && tiles_per_split >= kLongTiles) ? kLongStages : kShortStages, l2pf = 0;
  lc.dynamicSmemBytes = smem_bytes(ns);
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
  // fold depends on the model only (2G query rows with both flows), never
  // on which flows are active, so a row's arithmetic is the same either way
  const int fold = 2 * D.G <= 8 ? 1 : 0;
  cudaLaunchKernelEx(&lc, k_attn_tma, P.kv, (const float*)Bf.qatt, Bf.ctrl, (__nv_bfloat16*)Bf.o, R.B, D.Hkv, D.G,
                     Bf.kvm, layer, flo, fhi, ns, l2pf, fold);
}

}  // namespace df
