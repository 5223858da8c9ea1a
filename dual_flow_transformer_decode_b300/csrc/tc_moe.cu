// Grouped expert GEMMs of the MoE layer with router replay, on the tensor
// cores ("Mecanismos Clave", Replay de Router: the auxiliary flow reuses the
// experts the primary router chose and applies them with its own gates).
//
// After routing, every selected expert e has an entry list (token b, slot j)
// in ascending b.  k_moe_gather packs the expert's rows into one block:
// row 2i is the primary row and row 2i+1 the auxiliary row of its i-th entry.
// The gate/up and down GEMMs then run one CTA per (expert, 128-row weight
// tile) with N = 2 * entries (padded to 16) stacked rows, so each selected
// expert's weights are read from HBM once for both flows; CTAs of experts
// nobody selected exit at once.  Same tcgen05/TMEM/TMA pipeline as the dense
// GEMM, without K-splits (K = d or Fe gives each CTA 16-32 K blocks).
// Epilogues: gate/up -> SwiGLU with the b coupling (the primary partner of
// row 2i+1 is row 2i of the same tile); down -> raw expert outputs, combined
// per token in slot order by k_moe_combine_tc with both flows' gates and the
// c coupling.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdlib>

#include "ptx.cuh"
#include "tc_moe.h"

namespace df {

namespace {

// Ring depth.  Two stages (about 50 KB of shared memory at 64 stacked rows,
// four CTAs per SM) measured faster than four stages at two CTAs per SM:
// the MoE step 3.26 -> 3.21 ms, with the auxiliary fan-out 3.65 -> 3.49 ms;
// one stage (six CTAs per SM, no overlap inside a CTA) 3.84 ms.  The
// weight stream of one CTA is bound by its own load -> MMA -> release
// round trips, so more CTAs per SM stream more than deeper rings.
constexpr int kStages = 2;
constexpr int kBK = 64;
constexpr int kBM = 128;
constexpr int kStageW = kBM * kBK * 2;
constexpr int kXBox = 16;  // rows per activation TMA box

struct MoeArgs {
  const int* ecount;
  const int* elist;
  const float* bvec;
  Couple C;
  __nv_bfloat16* zE;  // [E][nxe][Fe]
  float* yE;          // [E][nxe][d]
  Ctrl* ctrl;
  int maxB, k, E, Fe, d, nxe;
  int B;          // batch: entries below B*k are replayed, the others auxiliary-own
  int prim, aux;  // active flows
  int op;         // 0: gate/up, 1: down
  int tiles;      // 128-row weight tiles per expert
  int rows_w;     // weight rows per expert (2Fe or d)
  int stages;     // ring depth
};

__global__ void __launch_bounds__(128, 1)
    k_tc_moe(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tx, int K, MoeArgs a) {
  const int e = blockIdx.x / a.tiles, tile = blockIdx.x % a.tiles;
  // Routing finished before the previous kernel's CTAs passed their own
  // dependency wait, which each of them does before it lets this grid
  // start, so the expert's entry count is final here (read from L2, not
  // through L1): CTAs of unselected experts leave at once and the others
  // request their first weight stages before the dependency resolves.
  const int cnt = __ldcg(a.ecount + e);
  if (cnt == 0) return;  // uniform across the CTA
  const int S = a.stages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int N = (2 * cnt + 15) / 16 * 16;
  const int stage_x = N * kBK * 2;
  uint8_t* sw = base;
  uint8_t* sx = base + S * kStageW;
  size_t region = (size_t)S * (kStageW + (size_t)a.nxe * kBK * 2);
  if ((size_t)a.nxe * kBM * 4 > region) region = (size_t)a.nxe * kBM * 4;
  uint64_t* full = reinterpret_cast<uint64_t*>(base + region);
  uint64_t* empty = full + S;
  uint64_t* done = empty + S;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* flags = reinterpret_cast<volatile int*>(tslot + 1);
  float* st = reinterpret_cast<float*>(base);  // [N][128] result tile, reuses the ring

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nk = K / kBK;
  const uint32_t ncols = N <= 32 ? 32 : N <= 64 ? 64 : N <= 128 ? 128 : 256;
  const int wrow = e * a.rows_w + tile * kBM, xrow = e * a.nxe;

  if (tid == 0) {
    ptx::prefetch_tmap(&tw);
    ptx::prefetch_tmap(&tx);
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(done, 1);
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
  ptx::grid_dep_launch();

  if (warp == 0 && lane == 0) {
    const uint64_t pol_w = ptx::policy_evict_first();
    // the weights do not depend on the previous kernel: the first stages'
    // weight tiles are requested before waiting for it
    const int pre = nk < S ? nk : S;
    for (int i = 0; i < pre; ++i) {
      ptx::mbar_arrive_expect_tx(&full[i], kStageW + stage_x);
      ptx::tma_load_2d_hint(sw + i * kStageW, &tw, &full[i], i * kBK, wrow, pol_w);
    }
    ptx::grid_dep_wait();
    for (int i = 0; i < pre; ++i)
      for (int q = 0; q < N / kXBox; ++q)
        ptx::tma_load_2d(sx + i * stage_x + q * kXBox * kBK * 2, &tx, &full[i], i * kBK, xrow + q * kXBox);
    for (int i = pre; i < nk; ++i) {
      const int s = i % S;
      if (!ptx::mbar_wait(&empty[s], ((i / S) - 1) & 1)) {
        flags[0] = 1;
        latch_error(a.ctrl, kErrTimeout, 300);
        break;
      }
      ptx::mbar_arrive_expect_tx(&full[s], kStageW + stage_x);
      ptx::tma_load_2d_hint(sw + s * kStageW, &tw, &full[s], i * kBK, wrow, pol_w);
      for (int q = 0; q < N / kXBox; ++q)
        ptx::tma_load_2d(sx + s * stage_x + q * kXBox * kBK * 2, &tx, &full[s], i * kBK, xrow + q * kXBox);
    }
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = ptx::idesc_bf16_f32(kBM, N);
    for (int i = 0; i < nk; ++i) {
      const int s = i % S;
      if (!ptx::mbar_wait(&full[s], (i / S) & 1)) {
        flags[0] = 1;
        latch_error(a.ctrl, kErrTimeout, 301);
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
  } else {
    ptx::grid_dep_wait();
  }
  __syncwarp();
  const bool ok = ptx::mbar_wait(done, 0);
  ptx::tc_fence_after();
  if (!ok && tid == 0) {
    flags[0] = 1;
    latch_error(a.ctrl, kErrTimeout, 302);
  }
  __syncthreads();
  const bool aborted = flags[0] != 0;
  if (!aborted) {
    const int r = warp * 32 + lane;
    for (int j0 = 0; j0 < N; j0 += 16) {
      float v[16];
      ptx::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + j0, v);
#pragma unroll
      for (int q = 0; q < 16; ++q) st[(j0 + q) * kBM + r] = v[q];
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (!aborted) {
    if (a.op == 0) {
      // SwiGLU over (entry i, pair p): gate = feature p, up = feature p + 64
      for (int u = tid; u < cnt * 64; u += 128) {
        const int i = u / 64, p = u % 64;
        const int fi = tile * 64 + p;
        const int ent = a.elist[(size_t)e * a.maxB + i];
        const bool own = ent >= a.B * a.k;  // auxiliary-own expert: no primary partner, no b coupling
        const float* r1 = st + (2 * i) * kBM;
        const float* r2 = st + (2 * i + 1) * kBM;
        const float z1 = silu_f(r1[p]) * r1[p + 64];
        if (a.prim && !own) {
          if (a.C.save) a.C.z1s[(size_t)ent * a.Fe + fi] = z1;
          a.zE[((size_t)e * a.nxe + 2 * i) * a.Fe + fi] = __float2bfloat16_rn(z1);
        }
        if (a.aux) {
          const float zp = own ? 0.f : a.C.saved ? a.C.z1s[(size_t)ent * a.Fe + fi] : z1;
          const float z2 = fmaf(a.bvec[fi], zp, silu_f(r2[p]) * r2[p + 64]);
          a.zE[((size_t)e * a.nxe + 2 * i + 1) * a.Fe + fi] = __float2bfloat16_rn(z2);
        }
      }
    } else {
      // raw expert outputs of the active rows
      for (int u = tid; u < 2 * cnt * kBM; u += 128) {
        const int m = u / kBM, n = u % kBM;
        const int f = m & 1;
        if ((f == 0 && !a.prim) || (f == 1 && !a.aux)) continue;
        a.yE[((size_t)e * a.nxe + m) * a.d + tile * kBM + n] = st[m * kBM + n];
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tmem, ncols);
}

// Pack the rows of each selected expert: row 2i <- primary row of entry i,
// row 2i+1 <- auxiliary row of entry i.
__global__ void k_moe_gather(const __nv_bfloat16* __restrict__ u, const int* __restrict__ ecount,
                             const int* __restrict__ elist, __nv_bfloat16* __restrict__ xg, int B, int d, int k,
                             int ka, int maxB, int nxe) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int e = blockIdx.x, slot = blockIdx.y;
  if (slot >= 2 * ecount[e]) return;
  const int ent = elist[(size_t)e * maxB + slot / 2];
  const int f = slot & 1;
  uint4* dst = reinterpret_cast<uint4*>(xg + ((size_t)e * nxe + slot) * d);
  if (ent >= B * k) {
    // auxiliary-own entry: only the auxiliary row exists; the primary slot
    // is zero, so its SwiGLU output, and the b coupling it feeds, is zero
    const int b = (ent - B * k) / (ka - k);
    if (f == 0) {
      for (int i = threadIdx.x; i < d / 8; i += blockDim.x) dst[i] = make_uint4(0u, 0u, 0u, 0u);
      return;
    }
    const uint4* src = reinterpret_cast<const uint4*>(u + (size_t)(B + b) * d);
    for (int i = threadIdx.x; i < d / 8; i += blockDim.x) dst[i] = src[i];
    return;
  }
  const int b = ent / k;
  const uint4* src = reinterpret_cast<const uint4*>(u + (size_t)(f * B + b) * d);
  for (int i = threadIdx.x; i < d / 8; i += blockDim.x) dst[i] = src[i];
}

// y_f = sum_j gate_f[j] * y_expert(e_j)[row of (b, j, f)] in slot order,
// y2 += c ⊙ y1, h += y.  CTA (stacked row, 256-feature chunk); the row's
// entries (expert, output row, gates) are staged in shared memory first.
constexpr int kCombineMaxK = 16;

__global__ void k_moe_combine_tc(const float* __restrict__ yE, const float* __restrict__ gate,
                                 const int* __restrict__ topk_l, const int* __restrict__ topkx,
                                 const int* __restrict__ eslot, const float* __restrict__ cvec,
                                 float* __restrict__ h, Couple C, int B, int lo, int d, int k, int ka, int nxe) {
  __shared__ size_t ofs[kCombineMaxK];  // start of the primary row of entry j in yE
  __shared__ float g_own[kCombineMaxK], g_prim[kCombineMaxK];
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int m = lo + blockIdx.x;
  const int f = m >= B, b = m - f * B;
  const int kr = f ? ka : k;  // entries of this row: the replayed ones, then the auxiliary-own ones
  if (threadIdx.x < kr) {
    const int j = threadIdx.x;
    if (j < k) {
      ofs[j] = ((size_t)topk_l[b * k + j] * nxe + 2 * eslot[b * k + j]) * d;
      g_prim[j] = gate[(size_t)b * ka + j];
    } else {
      const int jx = j - k, ent = B * k + b * (ka - k) + jx;
      ofs[j] = ((size_t)topkx[b * (ka - k) + jx] * nxe + 2 * eslot[ent]) * d;
    }
    g_own[j] = gate[(size_t)m * ka + j];
  }
  __syncthreads();
  const int n = blockIdx.y * blockDim.x + threadIdx.x;
  if (n >= d) return;
  float y = 0.f;
  for (int j = 0; j < kr; ++j) y = fmaf(g_own[j], yE[ofs[j] + (size_t)f * d + n], y);
  if (f) {
    float y1;
    if (C.saved) {
      y1 = C.y1s[(size_t)b * d + n];
    } else {
      y1 = 0.f;
      for (int j = 0; j < k; ++j) y1 = fmaf(g_prim[j], yE[ofs[j] + n], y1);
    }
    y = fmaf(cvec[n], y1, y);
  } else if (C.save) {
    C.y1s[(size_t)b * d + n] = y;
  }
  h[(size_t)m * d + n] += y;
}

// The combine of k_moe_combine_tc followed by the RMSNorm of the updated
// residual row with gains gn (the next layer's attention norm, or the final
// norm), in one launch: CTA m (256 threads) takes stacked row m, thread t the
// float4 groups t, t + 256, ... of the row, so every element's combine and
// the row's sum of squares are computed exactly as by the two separate
// kernels.
__global__ void __launch_bounds__(256) k_moe_combine_norm(
    const float* __restrict__ yE, const float* __restrict__ gate, const int* __restrict__ topk_l,
    const int* __restrict__ topkx, const int* __restrict__ eslot, const float* __restrict__ cvec,
    float* __restrict__ h, Couple C, int B, int lo, int d, int k, int ka, int nxe, const float* __restrict__ gn,
    __nv_bfloat16* __restrict__ u, float eps) {
  __shared__ size_t ofs[kCombineMaxK];
  __shared__ float g_own[kCombineMaxK], g_prim[kCombineMaxK];
  __shared__ float red[32];
  const int n4 = d >> 2;
  const float4* g4 = reinterpret_cast<const float4*>(gn);
  float4 gv[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int i = threadIdx.x + q * 256;
    if (i < n4) gv[q] = g4[i];
  }
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int m = lo + blockIdx.x;
  const int f = m >= B, b = m - f * B;
  const int kr = f ? ka : k;
  if (threadIdx.x < kr) {
    const int j = threadIdx.x;
    if (j < k) {
      ofs[j] = ((size_t)topk_l[b * k + j] * nxe + 2 * eslot[b * k + j]) * d;
      g_prim[j] = gate[(size_t)b * ka + j];
    } else {
      const int jx = j - k, ent = B * k + b * (ka - k) + jx;
      ofs[j] = ((size_t)topkx[b * (ka - k) + jx] * nxe + 2 * eslot[ent]) * d;
    }
    g_own[j] = gate[(size_t)m * ka + j];
  }
  __syncthreads();
  float4 v[8];
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int i = threadIdx.x + q * 256;
    if (i < n4) {
      const int n = 4 * i;
      float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j = 0; j < kr; ++j) {
        const float4 e = *reinterpret_cast<const float4*>(yE + ofs[j] + (size_t)f * d + n);
        const float gj = g_own[j];
        y = make_float4(fmaf(gj, e.x, y.x), fmaf(gj, e.y, y.y), fmaf(gj, e.z, y.z), fmaf(gj, e.w, y.w));
      }
      if (f) {
        float4 y1;
        if (C.saved) {
          y1 = *reinterpret_cast<const float4*>(C.y1s + (size_t)b * d + n);
        } else {
          y1 = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int j = 0; j < k; ++j) {
            const float4 e = *reinterpret_cast<const float4*>(yE + ofs[j] + n);
            const float gj = g_prim[j];
            y1 = make_float4(fmaf(gj, e.x, y1.x), fmaf(gj, e.y, y1.y), fmaf(gj, e.z, y1.z), fmaf(gj, e.w, y1.w));
          }
        }
        const float4 c = *reinterpret_cast<const float4*>(cvec + n);
        y = make_float4(fmaf(c.x, y1.x, y.x), fmaf(c.y, y1.y, y.y), fmaf(c.z, y1.z, y.z), fmaf(c.w, y1.w, y.w));
      } else if (C.save) {
        *reinterpret_cast<float4*>(C.y1s + (size_t)b * d + n) = y;
      }
      float4* hp = reinterpret_cast<float4*>(h + (size_t)m * d + n);
      float4 hv = *hp;
      hv.x += y.x;
      hv.y += y.y;
      hv.z += y.z;
      hv.w += y.w;
      *hp = hv;
      v[q] = hv;
      ss += v[q].x * v[q].x + v[q].y * v[q].y + v[q].z * v[q].z + v[q].w * v[q].w;
    }
  }
  ss = block_sum(ss, red);
  const float r = 1.0f / sqrtf(ss / (float)d + eps);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int i = threadIdx.x + q * 256;
    if (i < n4) {
      const float4 gg = gv[q];
      const float a = v[q].x * r * gg.x, bb = v[q].y * r * gg.y, c = v[q].z * r * gg.z, e = v[q].w * r * gg.w;
      __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(u + (size_t)m * d + 4 * i);
      o[0] = __floats2bfloat162_rn(a, bb);
      o[1] = __floats2bfloat162_rn(c, e);
    }
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
}

bool make_map(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t smem_bytes(int nxe, int stages) {
  size_t region = (size_t)stages * (kStageW + (size_t)nxe * kBK * 2);
  if ((size_t)nxe * kBM * 4 > region) region = (size_t)nxe * kBM * 4;
  return 1024 + region + 2 * (size_t)stages * 8 + 8 + 16;
}

}  // namespace

int moe_nxe(const Dims& D) { return (2 * D.maxB + 15) / 16 * 16; }

bool moe_tc_init(MoePlan& P, const Dims& D, const Buffers& Bf, const std::vector<const void*>& wgu,
                 const std::vector<const void*>& wd, std::string* err) {
  P.enabled = false;
  const char* e = getenv("DF_NO_TC");
  if (e && e[0] == '1') return true;
  if (!D.E || !D.bf16 || D.d % kBM || D.Fe % kBK) return true;  // gate/up tiles: Fe/64 (64 gate + 64 up rows)
  const int nxe = moe_nxe(D);
  const int st = kStages;
  if (nxe > 256 || smem_bytes(nxe, st) > 227 * 1024) return true;
  P.nxe = nxe;
  P.stages = st;
  P.w_gu.resize(D.L);
  P.w_d.resize(D.L);
  bool ok = true;
  for (int l = 0; l < D.L; ++l) {
    ok &= make_map(&P.w_gu[l], wgu[l], D.d, (uint64_t)D.E * 2 * D.Fe, kBM);
    ok &= make_map(&P.w_d[l], wd[l], D.Fe, (uint64_t)D.E * D.d, kBM);
  }
  ok &= make_map(&P.x_g, Bf.xg, D.d, (uint64_t)D.E * nxe, kXBox);
  ok &= make_map(&P.x_z, Bf.zEt, D.Fe, (uint64_t)D.E * nxe, kXBox);
  if (!ok) {
    if (err) *err = "cuTensorMapEncodeTiled failed for an expert matrix";
    return false;
  }
  cudaFuncSetAttribute(k_tc_moe, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes(nxe, kStages));
  P.enabled = true;
  return true;
}

void moe_tc_free(MoePlan& P) {
  P.w_gu.clear();
  P.w_d.clear();
  P.enabled = false;
}

void moe_tc_forward(const MoePlan& P, const Dims& D, const Buffers& Bf, int layer, const float* bvec,
                    const float* cvec, const Couple& C, const Rows& R, cudaStream_t s, const float* next_norm) {
  const int prim = R.has_primary(), aux = R.has_aux();
  launch_pdl(k_moe_gather, dim3(D.E, P.nxe), dim3(128), 0, s, (const __nv_bfloat16*)Bf.u, (const int*)Bf.ecount,
             (const int*)Bf.elist, (__nv_bfloat16*)Bf.xg, R.B, D.d, D.k, D.ka, D.maxB, P.nxe);
  MoeArgs a{};
  a.ecount = Bf.ecount;
  a.elist = Bf.elist;
  a.bvec = bvec;
  a.C = C;
  a.zE = (__nv_bfloat16*)Bf.zEt;
  a.yE = Bf.yEt;
  a.ctrl = Bf.ctrl;
  a.maxB = D.maxB;
  a.k = D.k;
  a.B = R.B;
  a.E = D.E;
  a.Fe = D.Fe;
  a.d = D.d;
  a.nxe = P.nxe;
  a.prim = prim;
  a.aux = aux;
  a.op = 0;
  a.tiles = 2 * D.Fe / kBM;
  a.rows_w = 2 * D.Fe;
  a.stages = P.stages;
  launch_pdl(k_tc_moe, dim3(D.E * a.tiles), dim3(128), smem_bytes(P.nxe, P.stages), s, P.w_gu[layer], P.x_g, D.d,
             a);
  a.op = 1;
  a.tiles = D.d / kBM;
  a.rows_w = D.d;
  launch_pdl(k_tc_moe, dim3(D.E * a.tiles), dim3(128), smem_bytes(P.nxe, P.stages), s, P.w_d[layer], P.x_z, D.Fe,
             a);
  const int* topk_l = Bf.topk + (size_t)layer * D.maxB * D.k;
  if (next_norm)
    launch_pdl(k_moe_combine_norm, dim3(R.hi - R.lo), dim3(256), 0, s, (const float*)Bf.yEt, (const float*)Bf.gate,
               topk_l, (const int*)Bf.topkx, (const int*)Bf.eslot, cvec, Bf.h, C, R.B, R.lo, D.d, D.k, D.ka, P.nxe,
               next_norm, (__nv_bfloat16*)Bf.u, D.eps);
  else
    launch_pdl(k_moe_combine_tc, dim3(R.hi - R.lo, (D.d + 255) / 256), dim3(256), 0, s, (const float*)Bf.yEt,
               (const float*)Bf.gate, topk_l, (const int*)Bf.topkx, (const int*)Bf.eslot, cvec, Bf.h, C, R.B, R.lo,
               D.d, D.k, D.ka, P.nxe);
}

}  // namespace df
