// Persistent decode-pass kernel for dense bf16 models (head_dim 128, G <= 4,
// at most 32 stacked rows): one launch runs every layer of a pass over the
// stacked rows, with the phases of "Arquitectura Central" and the couplings
// of "Mecanismos Clave" ("Resumen Técnico: Dual-Flow Transformers"):
//
//   per layer:  RMSNorm -> QKV (+ Q2 coupling, RoPE, cache append) ->
//               shared-KV attention -> Wo + residual -> RMSNorm ->
//               gate/up (+ SwiGLU, b coupling) -> down (+ c coupling, residual)
//
// Why one launch: at decode sizes every phase is a few microseconds of HBM
// streaming, and a kernel per phase pays a launch/dependency hand-off and a
// pipeline fill each time.  Here one CTA per SM runs a fixed, host-built list
// of tasks for the whole pass, and the weight and cache streams never stop at
// phase boundaries: nothing the producer warp loads depends on the step's
// activations.
//
// Warp roles (256 threads):
//   warp 0     weight/KV producer: every 128x64 weight k-block and 64-position
//              K or V tile of this CTA's tasks, in task order, by TMA into a
//              ring of 10 slots of 20 KB (16 KB weights/KV + 4 KB activations).
//   warp 1     MMA issuer: tcgen05.mma kind::f16, M = 128 weight rows, N =
//              stacked rows padded to 16, fp32 accumulators in two TMEM
//              buffers (a task's epilogue overlaps the next task's MMAs).
//              It also waits, in ring order, on every KV slot and hands it
//              to the compute warps, so each slot's "full" barrier has a
//              single waiter that sees all its phases (parity waits are only
//              sound then).
//   warp 2     activation producer: for each GEMM k-block, waits until the
//              rows it needs exist (counters in global memory) and loads them
//              by TMA beside the weights.
//   warps 4-7  compute: split-K reduction and the fused epilogues, RMSNorm
//              rows, shared-KV attention (mma.sync, as in the stand-alone
//              attention kernel), and the completion counters.
//
// Work split (host side, mk_batch): each GEMM phase is cut "stream-K" style
// into equal runs of (tile, k-block) units, one run per CTA; a tile's runs are
// its segments.  Segments write fp32 partial tiles; the last to arrive (a
// ticket) sums all of them in segment order and runs the epilogue, so results
// do not depend on arrival order.  Attention is cut into (sequence, KV head,
// KV range) segments merged the same way.  Dependencies only point to earlier
// phases and every role walks its CTA's list in order, so the pass cannot
// deadlock; every wait is bounded by %globaltimer and a CTA that gives up
// latches an error and makes the others stop.  The last CTA to finish zeroes
// the counters for the next launch.
//
// Status: opt-in (DF_MK=1).  It is correct (same parity cases as the kernel
// sequence) but at the dense1b_ctx1k decode shape it measured 2.6 ms per step
// against 1.12 ms for the per-layer kernels: every cross-CTA exchange here (a
// partial tile, an arrival count, a finished-tile count) is a round trip
// through L2 of about a microsecond, several per phase, where the cluster
// kernels exchange split-K partials through distributed shared memory and
// pay one launch hand-off per phase instead.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "mk_step.h"
#include "ptx.cuh"

namespace df {

namespace {

constexpr int kThreads = 256;
constexpr int kBM = 128;                    // weight rows per tile
constexpr int kBK = 64;                     // k elements per k-block
constexpr int kSlotW = kBM * kBK * 2;       // 16 KB: weight k-block or one K/V tile
constexpr int kMaxN = 32;
constexpr int kSlotX = kMaxN * kBK * 2;     // 4 KB: activation k-block (N rows)
constexpr int kSlot = kSlotW + kSlotX;      // 20 KB, a multiple of 1024
constexpr int kSlots = 10;
constexpr int kTP = 64;                     // positions per KV tile
constexpr int kHD = 128;
constexpr int kBox = kTP * 64 * 2;          // one 64-position x 64-dim TMA box
constexpr int kMaxRows = 8;                 // attention query rows per pair (2 flows x G <= 4)
constexpr int kApart = kMaxRows * (kHD + 2);  // floats per attention segment partial
constexpr int kMaxAttnSeg = 16;
constexpr size_t kScrBytes = 18432;         // reduced tile [128][N+1] / attention merge area
constexpr size_t kQsBytes = 16 * kHD * 2;   // attention queries [16][128] bf16
constexpr float kScale = 0.08838834764831845f;  // 1/sqrt(128)
constexpr uint64_t kWaitNs = 2000000000ull;

// Counter layout (uint32, zeroed between launches).
struct CntLayout {
  int L, MT, Hkv, maxB;
  // slices of tile t of phase ph in layer l that are finished
  __host__ __device__ size_t tile_done(int l, int ph, int t) const { return ((size_t)l * 4 + ph) * MT + t; }
  // segments of that tile whose partial is written
  __host__ __device__ size_t arr(int l, int ph, int t) const { return ((size_t)(L + l) * 4 + ph) * MT + t; }
  __host__ __device__ size_t phase_done(int l, int ph) const { return (size_t)L * 8 * MT + (size_t)l * 4 + ph; }
  __host__ __device__ size_t norm_done(int l, int w) const { return (size_t)L * 8 * MT + (size_t)L * 4 + l * 2 + w; }
  __host__ __device__ size_t attn_done(int l, int g) const {
    return (size_t)L * 8 * MT + (size_t)L * 6 + (size_t)l * Hkv + g;
  }
  __host__ __device__ size_t aticket(int pair) const {
    return (size_t)L * 8 * MT + (size_t)L * 6 + (size_t)L * Hkv + pair;
  }
  __host__ __device__ size_t cta_done() const { return aticket(0) + (size_t)maxB * Hkv; }
  __host__ __device__ size_t total() const { return cta_done() + 1; }
};

struct MkParams {
  const MkTask* tasks;
  const int* ntasks;
  int maxT;
  const CUtensorMap* wmap;   // [L][4]
  const CUtensorMap* xmap;   // [3]
  const CUtensorMap* kvmap;
  const MkLayer* layers;
  float* h;
  __nv_bfloat16* u;
  float* qatt;
  __nv_bfloat16* o;
  __nv_bfloat16* z;
  __nv_bfloat16* kv;
  const float* rope;
  Ctrl* ctrl;
  uint32_t* cnt;
  size_t ncnt;
  float* gpart;
  size_t gregion;
  float* apart;
  float *q1s, *z1s, *y1s;    // saved primary values, [L][maxB][...]
  CntLayout cl;
  const uint8_t* tnseg;      // [4][MT]: segments of each tile of each GEMM phase
  int d, qdim, kvdim, F, Hq, Hkv, G, maxB, max_len, B, lo, hi, N, save, saved;
  int segs_wo, segs_dn;      // segments of the Wo and down phases (tile slices finished per layer)
  float eps;
};

// ------------------------------------------------------------------ small helpers

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ticket_add(uint32_t* p) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
  return old;
}

// Release increment: this thread's earlier writes, and those of the CTA's
// threads ordered before it by a barrier, are visible at GPU scope before the
// counter moves.  `tma`: the data will also be read by TMA (the async proxy).
__device__ __forceinline__ void signal(uint32_t* c, bool tma = false) {
  if (tma) asm volatile("fence.proxy.async.global;" ::: "memory");
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(c) : "memory");
}

__device__ __forceinline__ void fence_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Named barrier of the four compute warps, and its AND-reduction form (every
// thread gets the same answer, so failure handling stays uniform).
__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool cbar_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// Gives up: stops this CTA's roles, tells the other CTAs, and (first error
// only) records where: CTA, task, what was awaited, target and value seen.
__device__ __noinline__ void raise_abort(volatile int* abort_s, Ctrl* ctrl, int code, int what = -1,
                                         uint32_t target = 0, uint32_t seen = 0) {
  *abort_s = 1;
  atomicExch(&ctrl->mk_abort, 1);
  if (atomicCAS(&ctrl->err, 0, kErrTimeout) == 0) {
    ctrl->err_info = code;
    ctrl->pad[0] = (int)blockIdx.x;
    ctrl->pad[1] = what;
    ctrl->pad[2] = (int)target;
    ctrl->pad[3] = (int)seen;
    ctrl->pad[4] = (int)threadIdx.x;
  }
}

__device__ __forceinline__ bool aborted(volatile int* abort_s, Ctrl* ctrl) {
  return *abort_s != 0 || *reinterpret_cast<volatile int*>(&ctrl->mk_abort) != 0;
}

// Spin until *c >= target (acquire); false after 2 s or when another CTA gave up.
// `what` identifies the counter (its index) in the error record.
__device__ bool wait_cnt(const uint32_t* c, uint32_t target, volatile int* abort_s, Ctrl* ctrl, int code, int what) {
  if (ld_acquire(c) >= target) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t it = 1;; ++it) {
    const uint32_t v = ld_acquire(c);
    if (v >= target) return true;
    if ((it & 15) == 0) {
      if (aborted(abort_s, ctrl)) return false;
      if (ptx::globaltimer() - t0 > kWaitNs) {
        raise_abort(abort_s, ctrl, code, what, target, v);
        return false;
      }
    }
  }
}

// KV tiles [i0, i1) of attention segment `seg` of `nseg`: the cache positions
// below t, split evenly; position t itself is handled by the last segment.
__host__ __device__ __forceinline__ void attn_range(int t, int seg, int nseg, int& i0, int& i1) {
  const int nt = (t + kTP - 1) / kTP;
  const int per = (nt + nseg - 1) / nseg;
  i0 = seg * per < nt ? seg * per : nt;
  i1 = i0 + per < nt ? i0 + per : nt;
}

__device__ __forceinline__ int task_slots(const MkTask& k, int t) {
  if (k.type == MK_GEMM) return k.a1 - k.a0;
  if (k.type == MK_ATTN) {
    int i0, i1;
    attn_range(t, k.seg, k.nseg, i0, i1);
    return 2 * (i1 - i0);
  }
  return 0;
}

// ------------------------------------------------------------------ mma.sync helpers (attention)

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
  __nv_bfloat162 hv = __floats2bfloat162_rn(x, y);
  float2 hf = __bfloat1622float2(hv);
  hi = *reinterpret_cast<uint32_t*>(&hv);
  lo = pack_bf16(x - hf.x, y - hf.y);
}

// Byte offset of (position, dim) in a K or V tile of two 128-byte-swizzled
// boxes (dims 0..63, 64..127).
__device__ __forceinline__ uint32_t sw_off(int pos, int dim) {
  const int box = dim >> 6, dd = dim & 63;
  return box * kBox + pos * 128 + ((((dd >> 3) ^ (pos & 7)) << 4)) + ((dd & 7) << 1);
}

__device__ __forceinline__ float bf16_bits_to_f(unsigned short x) {
  return __bfloat162float(__ushort_as_bfloat16(x));
}

// ------------------------------------------------------------------ producer warps

__device__ void role_w(const MkParams& p, const MkTask* tl, int nt, int t, uint8_t* ring, uint64_t* full,
                       uint64_t* empty, volatile int* abort_s) {
  const uint64_t pol = ptx::policy_evict_first();
  uint32_t q = 0;
  for (int i = 0; i < nt; ++i) {
    const MkTask k = tl[i];
    if (k.type == MK_GEMM) {
      const CUtensorMap* m = p.wmap + k.layer * 4 + k.phase;
      for (int kb = k.a0; kb < k.a1; ++kb, ++q) {
        const int s = q % kSlots;
        if (q >= kSlots && !ptx::mbar_wait(&empty[s], ((q / kSlots) - 1) & 1)) {
          raise_abort(abort_s, p.ctrl, 300, i, q);
          return;
        }
        if (*abort_s) return;
        ptx::mbar_arrive_expect_tx(&full[s], kSlotW);
        ptx::tma_load_2d_hint(ring + (size_t)s * kSlot, m, &full[s], kb * kBK, k.tile * kBM, pol);
      }
    } else if (k.type == MK_ATTN) {
      const int b = k.tile / p.Hkv, g = k.tile % p.Hkv;
      const int zK = ((k.layer * 2) * p.maxB + b) * p.Hkv + g, zV = zK + p.maxB * p.Hkv;
      int i0, i1;
      attn_range(t, k.seg, k.nseg, i0, i1);
      for (int it = i0; it < i1; ++it)
        for (int hv = 0; hv < 2; ++hv, ++q) {
          const int s = q % kSlots;
          if (q >= kSlots && !ptx::mbar_wait(&empty[s], ((q / kSlots) - 1) & 1)) {
            raise_abort(abort_s, p.ctrl, 301, i, q);
            return;
          }
          if (*abort_s) return;
          uint8_t* dst = ring + (size_t)s * kSlot;
          ptx::mbar_arrive_expect_tx(&full[s], kSlotW);
          ptx::tma_load_3d(dst, p.kvmap, &full[s], 0, it * kTP, hv ? zV : zK);
          ptx::tma_load_3d(dst + kBox, p.kvmap, &full[s], 64, it * kTP, hv ? zV : zK);
        }
    }
  }
}

__device__ void role_x(const MkParams& p, const MkTask* tl, int nt, int t, uint8_t* ring, uint64_t* full,
                       uint64_t* empty, volatile int* abort_s) {
  const uint32_t xbytes = (uint32_t)p.N * kBK * 2;
  const uint32_t M = (uint32_t)(p.hi - p.lo);
  uint32_t q = 0;
  for (int i = 0; i < nt; ++i) {
    const MkTask k = tl[i];
    if (k.type == MK_GEMM) {
      const CUtensorMap* m = p.xmap + (k.phase == MK_WO ? 1 : k.phase == MK_DN ? 2 : 0);
      bool dep_ok = false;
      for (int kb = k.a0; kb < k.a1; ++kb, ++q) {
        const int s = q % kSlots;
        if (q >= kSlots && !ptx::mbar_wait(&empty[s], ((q / kSlots) - 1) & 1)) {
          raise_abort(abort_s, p.ctrl, 310, i, q);
          return;
        }
        const uint32_t* c = nullptr;
        uint32_t target = 0;
        switch (k.phase) {
          case MK_QKV:
            if (!dep_ok) c = p.cnt + p.cl.norm_done(k.layer, 0), target = M;
            break;
          case MK_GU:
            if (!dep_ok) c = p.cnt + p.cl.norm_done(k.layer, 1), target = M;
            break;
          case MK_WO:  // o features [64 kb, 64 kb + 64) belong to head kb/2, KV group (kb/2)/G
            c = p.cnt + p.cl.attn_done(k.layer, (kb >> 1) / p.G), target = (uint32_t)p.B;
            break;
          default:     // MK_DN: z features of k-block kb come from gate/up tile kb
            c = p.cnt + p.cl.tile_done(k.layer, MK_GU, kb), target = p.tnseg[MK_GU * p.cl.MT + kb];
            break;
        }
        if (c) {
          if (!wait_cnt(c, target, abort_s, p.ctrl, 311, (int)(c - p.cnt))) return;
          dep_ok = true;
        }
        fence_async_global();
        ptx::mbar_arrive_expect_tx(&full[s], xbytes);
        ptx::tma_load_2d(ring + (size_t)s * kSlot + kSlotW, m, &full[s], kb * kBK, p.lo);
      }
    } else if (k.type == MK_ATTN) {
      const int n = task_slots(k, t);
      for (int j = 0; j < n; ++j, ++q) {
        const int s = q % kSlots;
        if (q >= kSlots && !ptx::mbar_wait(&empty[s], ((q / kSlots) - 1) & 1)) {
          raise_abort(abort_s, p.ctrl, 312, i, q);
          return;
        }
        ptx::mbar_arrive(&full[s]);
      }
    }
  }
}

__device__ void role_mma(const MkParams& p, const MkTask* tl, int nt, int t, uint8_t* ring, uint64_t* full,
                         uint64_t* empty, uint64_t* aready, uint64_t* accf, uint64_t* acce, uint32_t tmem,
                         volatile int* abort_s) {
  const uint32_t idesc = ptx::idesc_bf16_f32(kBM, p.N);
  uint32_t q = 0;
  int acc = 0;
  for (int i = 0; i < nt; ++i) {
    const MkTask k = tl[i];
    if (k.type == MK_GEMM) {
      const int buf = acc & 1, use = acc >> 1;
      ++acc;
      if (use > 0 && !ptx::mbar_wait(&acce[buf], (use - 1) & 1)) {
        raise_abort(abort_s, p.ctrl, 320, i, (uint32_t)acc);
        return;
      }
      ptx::tc_fence_after();
      const uint32_t d = tmem + (uint32_t)(buf * 32);
      for (int kb = k.a0; kb < k.a1; ++kb, ++q) {
        const int s = q % kSlots;
        if (!ptx::mbar_wait(&full[s], (q / kSlots) & 1)) {
          raise_abort(abort_s, p.ctrl, 321, i, q);
          return;
        }
        if (*abort_s) return;
        ptx::tc_fence_after();
        const uint32_t a0 = ptx::smem_u32(ring + (size_t)s * kSlot), b0 = a0 + kSlotW;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          ptx::mma_bf16(d, ptx::desc_sw128(a0 + kk * 32), ptx::desc_sw128(b0 + kk * 32), idesc,
                        (kb > k.a0 || kk > 0) ? 1u : 0u);
        ptx::mma_commit(&empty[s]);
      }
      ptx::mma_commit(&accf[buf]);
    } else {
      // KV slots: this thread observes every phase of every slot's full
      // barrier (a parity wait is only sound when no phase is skipped) and
      // hands each KV slot to the compute warps through its ready barrier.
      const int n = task_slots(k, t);
      for (int j = 0; j < n; ++j, ++q) {
        const int s = q % kSlots;
        if (!ptx::mbar_wait(&full[s], (q / kSlots) & 1)) {
          raise_abort(abort_s, p.ctrl, 322, i, q);
          return;
        }
        ptx::mbar_arrive(&aready[s]);
      }
    }
  }
}

// ------------------------------------------------------------------ compute warps

// Epilogue of pairs [p0, p1) of a finished 128-row tile; st[r * SP + m] =
// output feature n0 + r for stacked row lo + m.  Unit (sequence b, pair pp):
// features pp and pp + 64 (RoPE pair / gate-up pair) of the primary row b and
// the auxiliary row B + b, so the coupling partner of an auxiliary value is
// at hand.
// Row of pair pp in st: pp - rlo (first of the pair), pp + rhi (second).
__device__ void gemm_epilogue(const MkParams& p, const MkTask& k, int t, const float* st, int SP, int p0, int p1,
                              int rlo, int rhi) {
  const int ct = threadIdx.x - 128;
  const int B = p.B;
  const bool prim = p.lo < B, aux = p.hi > B;
  const int l = k.layer, n0 = k.tile * kBM;
  const MkLayer& Ly = p.layers[l];
  float* q1s = p.q1s + (size_t)l * p.maxB * p.qdim;
  float* z1s = p.z1s + (size_t)l * p.maxB * p.F;
  float* y1s = p.y1s + (size_t)l * p.maxB * p.d;
  const int np = p1 - p0;
  for (int un = ct; un < B * np; un += 128) {
    const int b = un / np, pp = p0 + un % np;
    float v1lo = 0.f, v1hi = 0.f, v2lo = 0.f, v2hi = 0.f;
    if (prim) {
      v1lo = st[(pp - rlo) * SP + b - p.lo];
      v1hi = st[(pp + rhi) * SP + b - p.lo];
    }
    if (aux) {
      v2lo = st[(pp - rlo) * SP + B + b - p.lo];
      v2hi = st[(pp + rhi) * SP + B + b - p.lo];
    }
    const int g0 = n0 + pp, g1 = g0 + 64;
    switch (k.phase) {
      case MK_QKV: {
        const float c = p.rope[(size_t)t * kHD + 2 * pp], sn = p.rope[(size_t)t * kHD + 2 * pp + 1];
        if (n0 < p.qdim) {
          if (prim) {
            if (p.save) {
              q1s[(size_t)b * p.qdim + g0] = v1lo;
              q1s[(size_t)b * p.qdim + g1] = v1hi;
            }
            p.qatt[(size_t)b * p.qdim + g0] = Num<__nv_bfloat16>::quant(v1lo * c - v1hi * sn);
            p.qatt[(size_t)b * p.qdim + g1] = Num<__nv_bfloat16>::quant(v1hi * c + v1lo * sn);
          }
          if (aux) {
            float q0 = v1lo, q1 = v1hi;
            if (p.saved) {
              q0 = q1s[(size_t)b * p.qdim + g0];
              q1 = q1s[(size_t)b * p.qdim + g1];
            }
            const float a0 = fmaf(Ly.a[g0], q0, v2lo), a1 = fmaf(Ly.a[g1], q1, v2hi);
            const size_t m = (size_t)(B + b) * p.qdim;
            p.qatt[m + g0] = Num<__nv_bfloat16>::quant(a0 * c - a1 * sn);
            p.qatt[m + g1] = Num<__nv_bfloat16>::quant(a1 * c + a0 * sn);
          }
        } else if (prim) {
          const bool isk = n0 < p.qdim + p.kvdim;
          const int g = (isk ? n0 - p.qdim : n0 - p.qdim - p.kvdim) / kHD;
          const size_t kvs = (size_t)p.maxB * p.Hkv * p.max_len * kHD;
          __nv_bfloat16* P =
              p.kv + ((size_t)l * 2 + (isk ? 0 : 1)) * kvs + (((size_t)b * p.Hkv + g) * p.max_len + t) * kHD;
          if (isk) {
            P[pp] = __float2bfloat16_rn(v1lo * c - v1hi * sn);
            P[pp + 64] = __float2bfloat16_rn(v1hi * c + v1lo * sn);
          } else {
            P[pp] = __float2bfloat16_rn(v1lo);
            P[pp + 64] = __float2bfloat16_rn(v1hi);
          }
        }
        break;
      }
      case MK_WO: {
        if (prim) {
          float* hp = p.h + (size_t)b * p.d;
          hp[g0] = __ldcg(hp + g0) + v1lo;
          hp[g1] = __ldcg(hp + g1) + v1hi;
        }
        if (aux) {
          float* hp = p.h + (size_t)(B + b) * p.d;
          hp[g0] = __ldcg(hp + g0) + v2lo;
          hp[g1] = __ldcg(hp + g1) + v2hi;
        }
        break;
      }
      case MK_GU: {
        const int fi = k.tile * 64 + pp;
        const float z1 = silu_f(v1lo) * v1hi;
        if (prim) {
          if (p.save) z1s[(size_t)b * p.F + fi] = z1;
          p.z[(size_t)b * p.F + fi] = __float2bfloat16_rn(z1);
        }
        if (aux) {
          const float zp = p.saved ? z1s[(size_t)b * p.F + fi] : z1;
          const float z2 = fmaf(Ly.b[fi], zp, silu_f(v2lo) * v2hi);
          p.z[(size_t)(B + b) * p.F + fi] = __float2bfloat16_rn(z2);
        }
        break;
      }
      default: {  // MK_DN
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int gn = kk ? g1 : g0;
          const float y1 = kk ? v1hi : v1lo, y2 = kk ? v2hi : v2lo;
          if (prim) {
            if (p.save) y1s[(size_t)b * p.d + gn] = y1;
            float* hp = p.h + (size_t)b * p.d + gn;
            *hp = __ldcg(hp) + y1;
          }
          if (aux) {
            const float yp = p.saved ? y1s[(size_t)b * p.d + gn] : y1;
            float* hp = p.h + (size_t)(B + b) * p.d + gn;
            *hp = __ldcg(hp) + fmaf(Ly.c[gn], yp, y2);
          }
        }
        break;
      }
    }
  }
}

// GEMM tasks are finished in two stages so that no CTA waits on a tile
// before it has posted all of its partials of the phase (a wait on the
// first tile before posting the second would chain the CTAs of a
// contiguous split one after another).
// Stage 1: accumulator -> registers; a tile with one segment is finished at
// once, otherwise the partial tile is written and the tile's arrival counter
// moves.
__device__ bool gemm_arrive(const MkParams& p, const MkTask& k, int t, uint64_t* accf, uint64_t* acce, int& acc,
                            uint32_t tmem, float* scr, volatile int* abort_s) {
  const int ct = threadIdx.x - 128, w = ct >> 5;
  const int buf = acc & 1, use = acc >> 1;
  ++acc;
  // warp-uniform before the warp-collective TMEM load
  const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait(&accf[buf], use & 1));
  ptx::tc_fence_after();
  float va[16], vb[16];
#pragma unroll
  for (int m = 0; m < 16; ++m) va[m] = vb[m] = 0.f;
  if (ok) {
    const uint32_t ta = tmem + ((uint32_t)(w * 32) << 16) + (uint32_t)(buf * 32);
    ptx::tmem_ld16(ta, va);
    if (p.N > 16) ptx::tmem_ld16(ta + 16, vb);
  }
  ptx::tc_fence_before();
  if (!cbar_and(ok)) {
    if (ct == 0) raise_abort(abort_s, p.ctrl, 330);
    return false;
  }
  if (ct == 0) ptx::mbar_arrive(&acce[buf]);
  const int N = p.N, SP = N + 1, r = ct;
  if (k.nseg == 1) {
    float* st = scr;
#pragma unroll
    for (int m = 0; m < kMaxN; ++m)
      if (m < N) st[r * SP + m] = m < 16 ? va[m] : vb[m - 16];
    cbar();
    gemm_epilogue(p, k, t, st, SP, 0, 64, 0, 64);
    cbar();
    if (ct == 0) {
      signal(p.cnt + p.cl.tile_done(k.layer, k.phase, k.tile), k.phase == MK_GU);
      signal(p.cnt + p.cl.phase_done(k.layer, k.phase));
    }
    return true;
  }
  float* mine = p.gpart + (size_t)k.phase * p.gregion + ((size_t)k.part * kBM + r) * N;
#pragma unroll
  for (int m = 0; m < kMaxN; m += 4)
    if (m < N) {
      const float4 x = m < 16 ? make_float4(va[m], va[m + 1], va[m + 2], va[m + 3])
                              : make_float4(vb[m - 16], vb[m - 15], vb[m - 14], vb[m - 13]);
      *reinterpret_cast<float4*>(mine + m) = x;
    }
  cbar();  // the signalling thread's release fence covers the whole CTA's stores
  if (ct == 0) signal(p.cnt + p.cl.arr(k.layer, k.phase, k.tile));
  return true;
}

// Stage 2 (tiles with several segments): once every segment of the tile has
// posted its partial, reduce this segment's slice of pairs over all segments
// in segment order (so no result depends on arrival order) and run the
// epilogue on it.  The slices of a tile's segments cover all 64 pairs.
__device__ bool gemm_finish(const MkParams& p, const MkTask& k, int t, float* scr, volatile int* abort_s) {
  const int ct = threadIdx.x - 128;
  bool okb = true;
  if (ct == 0)
    okb = wait_cnt(p.cnt + p.cl.arr(k.layer, k.phase, k.tile), k.nseg, abort_s, p.ctrl, 331,
                   (int)p.cl.arr(k.layer, k.phase, k.tile));
  if (!cbar_and(okb)) return false;
  const int N = p.N, SP = N + 1;
  const int p0 = k.seg * 64 / k.nseg, p1 = (k.seg + 1) * 64 / k.nseg, np = p1 - p0;
  const int E = 2 * np * N;        // slice elements: rows p0..p1-1 and 64+p0..64+p1-1, all columns
  const float* first = p.gpart + (size_t)k.phase * p.gregion + (size_t)(k.part - k.seg) * kBM * N;
  // Segments are staged through shared memory a chunk at a time, each chunk
  // with one round of loads; every element is summed in segment order.
  const int chunk = (int)(kScrBytes / 4) / E;
  float acc[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j] = 0.f;
  float4* stg4 = reinterpret_cast<float4*>(scr);
  for (int s0 = 0; s0 < k.nseg; s0 += chunk) {
    const int sc = min(chunk, k.nseg - s0), total = sc * (E / 4);
    for (int base = 0; base < total; base += 8 * 128) {
      // eight loads in flight per thread before any of them is stored
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int f4 = base + ct + u * 128;
        if (f4 < total) {
          const int sg = f4 / (E / 4), e = (f4 % (E / 4)) * 4;
          const int rr = e / N, m = e % N;
          const int row = rr < np ? p0 + rr : 64 + p0 + (rr - np);
          v[u] = __ldcg(reinterpret_cast<const float4*>(first + ((size_t)(s0 + sg) * kBM + row) * N + m));
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int f4 = base + ct + u * 128;
        if (f4 < total) stg4[f4] = v[u];
      }
    }
    cbar();
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int e = ct + j * 128;
      if (e < E)
        for (int sg = 0; sg < sc; ++sg) acc[j] += scr[sg * E + e];
    }
    cbar();
  }
  // compact slice tile: row rr (0..2np-1), column m at st[rr * SP + m]
  float* st = scr;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int e = ct + j * 128;
    if (e < E) st[(e / N) * SP + e % N] = acc[j];
  }
  cbar();
  gemm_epilogue(p, k, t, st, SP, p0, p1, p0, np - p0);
  cbar();
  if (ct == 0) {
    signal(p.cnt + p.cl.tile_done(k.layer, k.phase, k.tile), k.phase == MK_GU);
    signal(p.cnt + p.cl.phase_done(k.layer, k.phase));
  }
  return true;
}

__device__ bool norm_task(const MkParams& p, const MkTask& k, float* scr, volatile int* abort_s) {
  const int ct = threadIdx.x - 128, w = ct >> 5, lane = ct & 31;
  const int l = k.layer, m = k.tile, which = k.phase;
  bool ok = true;
  if (ct == 0) {
    if (which == 0 && l > 0)
      ok = wait_cnt(p.cnt + p.cl.phase_done(l - 1, MK_DN), (uint32_t)p.segs_dn, abort_s, p.ctrl, 340,
                    (int)p.cl.phase_done(l - 1, MK_DN));
    else if (which == 1)
      ok = wait_cnt(p.cnt + p.cl.phase_done(l, MK_WO), (uint32_t)p.segs_wo, abort_s, p.ctrl, 341,
                    (int)p.cl.phase_done(l, MK_WO));
  }
  if (!cbar_and(ok)) return false;
  const float4* hr = reinterpret_cast<const float4*>(p.h + (size_t)m * p.d);
  const float4* g4 = reinterpret_cast<const float4*>(which ? p.layers[l].g2 : p.layers[l].g1);
  const int n4 = p.d >> 2;  // <= 2048
  float4 x[16];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int i = ct + j * 128;
    if (i < n4) {
      x[j] = __ldcg(hr + i);
      ss += x[j].x * x[j].x + x[j].y * x[j].y + x[j].z * x[j].z + x[j].w * x[j].w;
    }
  }
  ss = warp_sum(ss);
  if (lane == 0) scr[w] = ss;
  cbar();
  const float tot = (scr[0] + scr[1]) + (scr[2] + scr[3]);
  const float r = 1.0f / sqrtf(tot / (float)p.d + p.eps);
  __nv_bfloat16* ur = p.u + (size_t)m * p.d;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int i = ct + j * 128;
    if (i < n4) {
      const float4 gg = g4[i];
      __nv_bfloat162 lo2 = __floats2bfloat162_rn(x[j].x * r * gg.x, x[j].y * r * gg.y);
      __nv_bfloat162 hi2 = __floats2bfloat162_rn(x[j].z * r * gg.z, x[j].w * r * gg.w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo2);
      pk.y = *reinterpret_cast<uint32_t*>(&hi2);
      *reinterpret_cast<uint2*>(ur + 4 * i) = pk;
    }
  }
  cbar();
  if (ct == 0) signal(p.cnt + p.cl.norm_done(l, which), true);
  return true;
}

// `apar` bit s: parity of the next KV hand-over of ring slot s.
__device__ bool attn_task(const MkParams& p, const MkTask& k, int t, uint8_t* ring, uint64_t* aready,
                          uint64_t* empty, uint32_t& q, uint32_t& apar, float* scr, __nv_bfloat16* qs, int* bc,
                          volatile int* abort_s) {
  const int ct = threadIdx.x - 128, w = ct >> 5, lane = ct & 31;
  const int l = k.layer, b = k.tile / p.Hkv, g = k.tile % p.Hkv;
  const int G = p.G, B = p.B;
  const int flo = p.lo / B, R = ((p.hi - p.lo) / B) * G;  // query rows, <= 8
  // the group's Q tiles and this step's K and V tiles must be finished
  bool ok = true;
  if (ct == 0) {
    for (int j = 0; j < G && ok; ++j)
      ok = wait_cnt(p.cnt + p.cl.tile_done(l, MK_QKV, g * G + j), p.tnseg[g * G + j], abort_s, p.ctrl, 350,
                    (int)p.cl.tile_done(l, MK_QKV, g * G + j));
    if (ok)
      ok = wait_cnt(p.cnt + p.cl.tile_done(l, MK_QKV, p.Hq + g), p.tnseg[p.Hq + g], abort_s, p.ctrl, 351,
                    (int)p.cl.tile_done(l, MK_QKV, p.Hq + g));
    if (ok)
      ok = wait_cnt(p.cnt + p.cl.tile_done(l, MK_QKV, p.Hq + p.Hkv + g), p.tnseg[p.Hq + p.Hkv + g], abort_s,
                    p.ctrl, 352,
                    (int)p.cl.tile_done(l, MK_QKV, p.Hq + p.Hkv + g));
  }
  if (!cbar_and(ok)) return false;

  float* ow = scr;                // [4][8][128] warp partial outputs
  float* mw = scr + 4 * 8 * kHD;  // [4][8]
  float* lw = mw + 32;            // [4][8]
  float* mt = lw + 32;            // [8] score of position t
  float* kt = mt + 8;             // [128] K and V at position t
  float* vt = kt + kHD;
  const bool has_t = k.seg == k.nseg - 1;

  // query rows (bf16 values) -> qs[16][128]; rows >= R are zero
  for (int idx = ct; idx < 16 * (kHD / 4); idx += 128) {
    const int r = idx >> 5, i4 = idx & 31;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < R) {
      const int f = flo + r / G, j = r % G;
      v = __ldcg(reinterpret_cast<const float4*>(p.qatt + (size_t)(f * B + b) * p.qdim + (g * G + j) * kHD) + i4);
    }
    __nv_bfloat162* dq = reinterpret_cast<__nv_bfloat162*>(qs + r * kHD + 4 * i4);
    dq[0] = __floats2bfloat162_rn(v.x, v.y);
    dq[1] = __floats2bfloat162_rn(v.z, v.w);
  }
  if (has_t) {
    const size_t kvs = (size_t)p.maxB * p.Hkv * p.max_len * kHD;
    const __nv_bfloat16* K = p.kv + ((size_t)l * 2) * kvs + (((size_t)b * p.Hkv + g) * p.max_len + t) * kHD;
    const __nv_bfloat16* V = K + kvs;
    kt[ct] = bf16_bits_to_f(__ldcg(reinterpret_cast<const unsigned short*>(K) + ct));
    vt[ct] = bf16_bits_to_f(__ldcg(reinterpret_cast<const unsigned short*>(V) + ct));
  }
  cbar();
  if (has_t) {
    for (int r = w; r < R; r += 4) {
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) acc = fmaf(__bfloat162float(qs[r * kHD + lane * 4 + e]), kt[lane * 4 + e], acc);
      acc = warp_sum(acc);
      if (lane == 0) mt[r] = acc * kScale;
    }
  }

  // ---- cache tiles below t: four warps x 16 positions per 64-position tile
  int i0, i1;
  attn_range(t, k.seg, k.nseg, i0, i1);
  const int gq = lane >> 2, tq = lane & 3;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  uint32_t qa[8][4];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const __nv_bfloat16* q0 = qs + gq * kHD + kk * 16 + 2 * tq;
    const __nv_bfloat16* q1 = qs + (gq + 8) * kHD + kk * 16 + 2 * tq;
    qa[kk][0] = *reinterpret_cast<const uint32_t*>(q0);
    qa[kk][1] = *reinterpret_cast<const uint32_t*>(q1);
    qa[kk][2] = *reinterpret_cast<const uint32_t*>(q0 + 8);
    qa[kk][3] = *reinterpret_cast<const uint32_t*>(q1 + 8);
  }
  const int mq = lane >> 3, r8 = lane & 7;
  for (int it = i0; it < i1; ++it) {
    const int sK = q % kSlots;
    ++q;
    const int sV = q % kSlots;
    ++q;
    const uint32_t parK = (apar >> sK) & 1u;
    apar ^= 1u << sK;
    const uint32_t parV = (apar >> sV) & 1u;
    apar ^= 1u << sV;
    // warp-uniform before the warp-collective ldmatrix / mma.sync
    const bool okw =
        __all_sync(0xffffffffu, ptx::mbar_wait(&aready[sK], parK) && ptx::mbar_wait(&aready[sV], parV));
    if (okw) {
      const uint32_t kbase = ptx::smem_u32(ring + (size_t)sK * kSlot);
      const uint32_t vbase = ptx::smem_u32(ring + (size_t)sV * kSlot);
      float sc[2][4];
#pragma unroll
      for (int nt2 = 0; nt2 < 2; ++nt2) sc[nt2][0] = sc[nt2][1] = sc[nt2][2] = sc[nt2][3] = 0.f;
      const int kpos = w * 16 + (mq >> 1) * 8 + r8;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t b00, b01, b10, b11;
        ldsm_x4(kbase + sw_off(kpos, kk * 16 + (mq & 1) * 8), b00, b01, b10, b11);
        mma_16816(sc[0], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b00, b01);
        mma_16816(sc[1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b10, b11);
      }
      const int pbase = it * kTP + w * 16 + 2 * tq;
      float corr[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float v[4];
#pragma unroll
        for (int nt2 = 0; nt2 < 2; ++nt2)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int pos = pbase + nt2 * 8 + e;
            v[nt2 * 2 + e] = pos < t ? sc[nt2][2 * hh + e] * kScale : -INFINITY;
          }
        float mx = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mo = m_run[hh], mn = fmaxf(mo, mx);
        corr[hh] = (mo == -INFINITY) ? 0.f : expf(mo - mn);
        float sum = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[e] = (v[e] == -INFINITY) ? 0.f : expf(v[e] - mn);
          sum += v[e];
        }
        m_run[hh] = mn;
        l_run[hh] = l_run[hh] * corr[hh] + sum;
#pragma unroll
        for (int nt2 = 0; nt2 < 2; ++nt2) {
          sc[nt2][2 * hh] = v[nt2 * 2];
          sc[nt2][2 * hh + 1] = v[nt2 * 2 + 1];
        }
      }
      uint32_t ph[4], pl[4];
      split_pair(sc[0][0], sc[0][1], ph[0], pl[0]);
      split_pair(sc[0][2], sc[0][3], ph[1], pl[1]);
      split_pair(sc[1][0], sc[1][1], ph[2], pl[2]);
      split_pair(sc[1][2], sc[1][3], ph[3], pl[3]);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        o[j][0] *= corr[0];
        o[j][1] *= corr[0];
        o[j][2] *= corr[1];
        o[j][3] *= corr[1];
      }
      const int vpos = w * 16 + (mq & 1) * 8 + r8;
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
    if (!cbar_and(okw)) {
      if (ct == 0) raise_abort(abort_s, p.ctrl, 353);
      return false;
    }
    if (ct == 0) {
      ptx::mbar_arrive(&empty[sK]);
      ptx::mbar_arrive(&empty[sV]);
    }
  }
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 1);
    l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 2);
  }
  // ---- warp partials of the R rows (rows gq < 8; rows gq + 8 are padding)
  if (gq < R) {
    if (tq == 0) {
      mw[w * 8 + gq] = m_run[0];
      lw[w * 8 + gq] = l_run[0];
    }
#pragma unroll
    for (int j = 0; j < 16; ++j)
      *reinterpret_cast<float2*>(ow + (w * 8 + gq) * kHD + j * 8 + 2 * tq) = make_float2(o[j][0], o[j][1]);
  }
  cbar();
  // ---- merge the warps (and position t): thread ct owns dim ct of every row
  const int i = ct;
  float Mr[kMaxRows], Lr[kMaxRows], Or[kMaxRows];
#pragma unroll
  for (int r = 0; r < kMaxRows; ++r) {
    Mr[r] = -INFINITY;
    Lr[r] = 0.f;
    Or[r] = 0.f;
    if (r < R) {
      float M = -INFINITY;
#pragma unroll
      for (int ww = 0; ww < 4; ++ww) M = fmaxf(M, mw[ww * 8 + r]);
      if (has_t) M = fmaxf(M, mt[r]);
      float acc = 0.f, den = 0.f;
#pragma unroll
      for (int ww = 0; ww < 4; ++ww) {
        const float mv = mw[ww * 8 + r];
        const float e = (mv == -INFINITY) ? 0.f : expf(mv - M);
        acc = fmaf(e, ow[(ww * 8 + r) * kHD + i], acc);
        den = fmaf(e, lw[ww * 8 + r], den);
      }
      if (has_t) {
        const float e = expf(mt[r] - M);
        acc = fmaf(e, vt[i], acc);
        den += e;
      }
      Mr[r] = M;
      Lr[r] = den;
      Or[r] = acc;
    }
  }
  if (k.nseg == 1) {
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r)
      if (r < R) {
        const int f = flo + r / G, j = r % G;
        p.o[(size_t)(f * B + b) * p.qdim + (g * G + j) * kHD + i] = __float2bfloat16_rn(Or[r] / Lr[r]);
      }
  } else {
    float* P = p.apart + (size_t)k.part * kApart;
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r)
      if (r < R) {
        P[r * (kHD + 2) + 2 + i] = Or[r];
        if (i == 0) {
          P[r * (kHD + 2)] = Mr[r];
          P[r * (kHD + 2) + 1] = Lr[r];
        }
      }
    cbar();  // the ticket's release covers the whole CTA's stores
    if (ct == 0) bc[0] = ((ticket_add(p.cnt + p.cl.aticket(k.tile)) + 1) % k.nseg) == 0;
    cbar();
    if (!bc[0]) return true;
    // last segment: merge all segments' partials in segment order; the
    // running max and sum of every (segment, row) first, in one round
    const float* P0 = p.apart + (size_t)(k.part - k.seg) * kApart;
    float* ml = scr;  // [nseg][8][2]
    for (int idx = ct; idx < k.nseg * kMaxRows; idx += 128) {
      const int sg = idx / kMaxRows, r = idx % kMaxRows;
      if (r < R) {
        const float2 v = make_float2(__ldcg(P0 + (size_t)sg * kApart + r * (kHD + 2)),
                                     __ldcg(P0 + (size_t)sg * kApart + r * (kHD + 2) + 1));
        reinterpret_cast<float2*>(ml)[idx] = v;
      }
    }
    cbar();
    float M[kMaxRows], den[kMaxRows], acc[kMaxRows];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      M[r] = -INFINITY;
      den[r] = 0.f;
      acc[r] = 0.f;
      if (r < R)
        for (int sg = 0; sg < k.nseg; ++sg) M[r] = fmaxf(M[r], ml[2 * (sg * kMaxRows + r)]);
    }
    for (int s0 = 0; s0 < k.nseg; s0 += 4) {
      float ov[kMaxRows][4];
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          ov[r][j] = (r < R && s0 + j < k.nseg) ? __ldcg(P0 + (size_t)(s0 + j) * kApart + r * (kHD + 2) + 2 + i) : 0.f;
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int sg = s0 + j;
          if (r < R && sg < k.nseg) {
            const float ms = ml[2 * (sg * kMaxRows + r)];
            if (ms != -INFINITY) {
              const float e = expf(ms - M[r]);
              den[r] = fmaf(e, ml[2 * (sg * kMaxRows + r) + 1], den[r]);
              acc[r] = fmaf(e, ov[r][j], acc[r]);
            }
          }
        }
    }
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r)
      if (r < R) {
        const int f = flo + r / G, j = r % G;
        p.o[(size_t)(f * B + b) * p.qdim + (g * G + j) * kHD + i] = __float2bfloat16_rn(acc[r] / den[r]);
      }
  }
  cbar();
  if (ct == 0) signal(p.cnt + p.cl.attn_done(l, g), true);
  return true;
}

__device__ void role_compute(const MkParams& p, const MkTask* tl, int nt, int t, uint8_t* ring, uint64_t* aready,
                             uint64_t* empty, uint64_t* accf, uint64_t* acce, uint32_t tmem, float* scr,
                             __nv_bfloat16* qs, int* bc, volatile int* abort_s) {
  uint32_t q = 0, apar = 0;
  int acc = 0;
  for (int i = 0; i < nt;) {
    const MkTask k = tl[i];
    bool ok = true;
    if (k.type == MK_GEMM) {
      // the run of this CTA's tasks in the same GEMM phase of the same layer
      int j = i + 1;
      while (j < nt && tl[j].type == MK_GEMM && tl[j].layer == k.layer && tl[j].phase == k.phase) ++j;
      for (int x = i; x < j && ok; ++x) {
        ok = gemm_arrive(p, tl[x], t, accf, acce, acc, tmem, scr, abort_s);
        q += tl[x].a1 - tl[x].a0;
      }
      for (int x = i; x < j && ok; ++x)
        if (tl[x].nseg > 1) ok = gemm_finish(p, tl[x], t, scr, abort_s);
      i = j;
    } else {
      if (k.type == MK_ATTN)
        ok = attn_task(p, k, t, ring, aready, empty, q, apar, scr, qs, bc, abort_s);
      else
        ok = norm_task(p, k, scr, abort_s);
      ++i;
    }
    if (!ok) return;
  }
}

__global__ void __launch_bounds__(kThreads, 1) k_mk_step(const __grid_constant__ MkParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = base;
  float* scr = reinterpret_cast<float*>(ring + (size_t)kSlots * kSlot);
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(reinterpret_cast<uint8_t*>(scr) + kScrBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(qs) + kQsBytes);
  uint64_t* empty = full + kSlots;
  uint64_t* aready = empty + kSlots;
  uint64_t* accf = aready + kSlots;
  uint64_t* acce = accf + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(acce + 2);
  volatile int* abort_s = reinterpret_cast<volatile int*>(tslot + 1);
  int* bc = reinterpret_cast<int*>(tslot + 2);  // [2]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const MkTask* tl = p.tasks + (size_t)blockIdx.x * p.maxT;
  const int nt = p.ntasks[blockIdx.x];
  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      ptx::mbar_init(&full[i], 2);  // the weight/KV producer and the activation producer
      ptx::mbar_init(&empty[i], 1);
      ptx::mbar_init(&aready[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&accf[i], 1);
      ptx::mbar_init(&acce[i], 1);
    }
    *abort_s = 0;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tslot, 64);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tslot;
  ptx::grid_dep_wait();
  const int t = *reinterpret_cast<volatile int*>(&p.ctrl->t);

  if (warp == 0) {
    if (lane == 0) role_w(p, tl, nt, t, ring, full, empty, abort_s);
  } else if (warp == 1) {
    if (lane == 0) role_mma(p, tl, nt, t, ring, full, empty, aready, accf, acce, tmem, abort_s);
  } else if (warp == 2) {
    if (lane == 0) role_x(p, tl, nt, t, ring, full, empty, abort_s);
  } else if (warp >= 4) {
    role_compute(p, tl, nt, t, ring, aready, empty, accf, acce, tmem, scr, qs, bc, abort_s);
  }
  __syncwarp();
  if (*abort_s) {
    // after giving up, let copies and MMAs already issued land before the
    // shared memory and TMEM are released
    const uint64_t t0 = ptx::globaltimer();
    while (ptx::globaltimer() - t0 < 1000000ull) {
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, 64);
  ptx::grid_dep_launch();
  if (tid == 0) {
    __threadfence();
    bc[1] = atomicAdd(p.cnt + p.cl.cta_done(), 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (bc[1]) {
    // every other CTA has finished: reset the counters for the next launch
    __threadfence();
    for (size_t i = tid; i < p.ncnt; i += kThreads) p.cnt[i] = 0;
    if (tid == 0) p.ctrl->mk_abort = 0;
  }
}

size_t smem_total() { return 1024 + (size_t)kSlots * kSlot + kScrBytes + kQsBytes + (3 * kSlots + 4) * 8 + 64; }

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

bool map2d(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int mpad_of(const Dims& D) { return (2 * D.maxB + 15) / 16 * 16; }
int max_tiles(const Dims& D) { return std::max({D.qkvn / kBM, D.d / kBM, 2 * D.F / kBM}); }
int max_rows(const Dims& D) { return std::min(2 * D.maxB, 2 * 16); }

// Generous bound on the tasks of one CTA (any batch the kernel supports).
int maxT_bound(const Dims& D) {
  const int S = D.sms;
  const int M = max_rows(D);
  auto gem = [&](int T, int KB) { return (T * KB) / (S * KB) + 3; };
  const int pairs = std::min(D.maxB, 16) * D.Hkv;
  const int per_layer = 2 * (M / S + 2) + gem(D.qkvn / kBM, D.d / kBK) + gem(D.d / kBM, D.qdim / kBK) +
                        gem(2 * D.F / kBM, D.d / kBK) + gem(D.d / kBM, D.F / kBK) + (pairs * kMaxAttnSeg) / S + 2;
  return D.L * per_layer + 8;
}

struct Region {
  size_t wmap, kvmap, xmap, layers, tnseg, ntasks, tasks, cnt, gpart, apart, total;
  size_t gregion, ncnt;
  int maxT;
};

Region region_of(const Dims& D) {
  Region g{};
  size_t cur = 0;
  auto take = [&](size_t bytes, size_t align) {
    cur = (cur + align - 1) / align * align;
    size_t o = cur;
    cur += bytes;
    return o;
  };
  const int S = D.sms, MT = max_tiles(D);
  g.maxT = maxT_bound(D);
  g.wmap = take((size_t)D.L * 4 * sizeof(CUtensorMap), 128);
  g.kvmap = take(sizeof(CUtensorMap), 128);
  g.xmap = take(3 * 3 * sizeof(CUtensorMap), 128);
  g.layers = take((size_t)D.L * sizeof(MkLayer), 64);
  g.tnseg = take(4 * (size_t)MT, 64);
  g.ntasks = take(3 * (size_t)S * 4, 64);
  g.tasks = take(3 * (size_t)S * g.maxT * sizeof(MkTask), 64);
  CntLayout cl{D.L, MT, D.Hkv, D.maxB};
  g.ncnt = cl.total();
  g.cnt = take(g.ncnt * 4, 256);
  g.gregion = (size_t)(MT + S) * kBM * kMaxN;
  g.gpart = take(4 * g.gregion * 4, 256);
  g.apart = take(mk_attn_partial_floats(D) * 4, 256);
  g.total = cur;
  return g;
}

// Segments per tile of the stream-K split below.
std::vector<int> streamk_nseg(int T, int KB, int S) {
  const long U = (long)T * KB;
  std::vector<int> n(T, 0);
  for (int c = 0; c < S; ++c) {
    long u0 = U * c / S, u1 = U * (c + 1) / S;
    while (u0 < u1) {
      const int tile = (int)(u0 / KB);
      n[tile] += 1;
      u0 = std::min(u1, (long)(tile + 1) * KB);
    }
  }
  return n;
}

// Stream-K split of one GEMM phase: CTA c takes units [U c / S, U (c+1) / S)
// of the (tile, k-block) sequence; a run inside one tile is a segment.
void add_gemm_phase(std::vector<std::vector<MkTask>>& lists, int layer, int phase, int T, int KB, int S) {
  const long U = (long)T * KB;
  std::vector<std::vector<int>> seg_cta(T), seg_a0(T), seg_a1(T);
  for (int c = 0; c < S; ++c) {
    long u0 = U * c / S, u1 = U * (c + 1) / S;
    while (u0 < u1) {
      const int tile = (int)(u0 / KB);
      const long e = std::min(u1, (long)(tile + 1) * KB);
      seg_cta[tile].push_back(c);
      seg_a0[tile].push_back((int)(u0 - (long)tile * KB));
      seg_a1[tile].push_back((int)(e - (long)tile * KB));
      u0 = e;
    }
  }
  uint32_t part = 0;
  for (int tile = 0; tile < T; ++tile) {
    const int ns = (int)seg_cta[tile].size();
    for (int s = 0; s < ns; ++s) {
      MkTask k{};
      k.type = MK_GEMM;
      k.phase = (uint8_t)phase;
      k.layer = (uint16_t)layer;
      k.tile = (uint16_t)tile;
      k.a0 = (uint16_t)seg_a0[tile][s];
      k.a1 = (uint16_t)seg_a1[tile][s];
      k.seg = (uint8_t)s;
      k.nseg = (uint8_t)ns;
      k.part = part + s;
      lists[seg_cta[tile][s]].push_back(k);
    }
    part += ns;
  }
}

void add_norm_phase(std::vector<std::vector<MkTask>>& lists, int layer, int which, int lo, int hi, int S) {
  const int M = hi - lo;
  for (int j = 0; j < M; ++j) {
    MkTask k{};
    k.type = MK_NORM;
    k.phase = (uint8_t)which;
    k.layer = (uint16_t)layer;
    k.tile = (uint16_t)(lo + j);
    const int c = (int)(((long)j * S / M + (which ? S / 2 : 0)) % S);
    lists[c].push_back(k);
  }
}

void add_attn_phase(std::vector<std::vector<MkTask>>& lists, int layer, int B, int Hkv, int S) {
  const int pairs = B * Hkv;
  const int nseg = std::max(1, std::min(kMaxAttnSeg, S / pairs));
  const int ntask = pairs * nseg;
  for (int i = 0; i < ntask; ++i) {
    MkTask k{};
    k.type = MK_ATTN;
    k.layer = (uint16_t)layer;
    k.tile = (uint16_t)(i / nseg);
    k.seg = (uint8_t)(i % nseg);
    k.nseg = (uint8_t)nseg;
    k.part = (uint32_t)i;
    lists[(int)((long)i * S / ntask)].push_back(k);
  }
}

}  // namespace

namespace {
// Whether the model has the shapes the kernel handles (the workspace region
// is reserved for every such model, whether or not the kernel is enabled).
bool mk_eligible(const Dims& D, std::string* why) {
  auto no = [&](const char* m) {
    if (why) *why = m;
    return false;
  };
  if (!D.bf16) return no("not bf16");
  if (D.E) return no("MoE model");
  if (D.paged) return no("paged KV cache");
  if (D.hd != kHD) return no("head_dim is not 128");
  if (D.G > 4) return no("more than 4 query heads per KV head");
  if (D.d % kBM || D.d > 8192) return no("d_model not a multiple of 128 (or above 8192)");
  if (D.F % kBK || D.F <= 0) return no("ffn_hidden not a multiple of 64");
  if (D.sms <= 0 || D.sms > 255) return no("SM count outside 1..255");
  if (max_tiles(D) > 65535 || D.L > 65535) return no("too many tiles");
  return true;
}
}  // namespace

bool mk_supported(const Dims& D, std::string* why) {
  if (!mk_eligible(D, why)) return false;
  // Opt-in: measured slower than the per-layer kernel sequence at the
  // dense1b_ctx1k decode shape (its cross-CTA reductions and dependency
  // polls each cost an L2 round trip, where the cluster kernels use
  // distributed shared memory).
  const char* e = getenv("DF_MK");
  if (!(e && e[0] == '1')) {
    if (why) *why = "not enabled (DF_MK=1)";
    return false;
  }
  if (!encode_fn()) {
    if (why) *why = "no cuTensorMapEncodeTiled";
    return false;
  }
  return true;
}

size_t mk_workspace_bytes(const Dims& D) {
  if (!mk_eligible(D, nullptr)) return 0;
  return region_of(D).total;
}

bool mk_init(MkPlan& P, const Dims& D, const Buffers& Bf, void* region, void* kv,
             const std::vector<const void*>& wqkv, const std::vector<const void*>& wo,
             const std::vector<const void*>& wgu, const std::vector<const void*>& wd,
             const std::vector<const float*>& g1, const std::vector<const float*>& g2,
             const std::vector<const float*>& a, const std::vector<const float*>& b,
             const std::vector<const float*>& c, cudaStream_t s, std::string* err) {
  (void)Bf;
  P = MkPlan{};
  if (!region || !mk_supported(D, nullptr)) return true;
  const Region g = region_of(D);
  char* base = static_cast<char*>(region);
  P.sms = D.sms;
  P.max_tiles = max_tiles(D);
  P.maxT_cap = g.maxT;
  P.wmap = reinterpret_cast<CUtensorMap*>(base + g.wmap);
  P.kvmap = reinterpret_cast<CUtensorMap*>(base + g.kvmap);
  P.layers = reinterpret_cast<MkLayer*>(base + g.layers);
  P.tnseg = reinterpret_cast<uint8_t*>(base + g.tnseg);
  P.cnt = reinterpret_cast<uint32_t*>(base + g.cnt);
  P.ncnt = g.ncnt;
  P.gpart = reinterpret_cast<float*>(base + g.gpart);
  P.gregion = g.gregion;
  P.apart = reinterpret_cast<float*>(base + g.apart);
  for (int r = 0; r < 3; ++r) {
    P.rs[r].xmap = reinterpret_cast<CUtensorMap*>(base + g.xmap) + 3 * r;
    P.rs[r].ntasks = reinterpret_cast<int*>(base + g.ntasks) + (size_t)r * D.sms;
    P.rs[r].tasks = reinterpret_cast<MkTask*>(base + g.tasks) + (size_t)r * D.sms * g.maxT;
    P.rs[r].maxT = g.maxT;
  }
  std::vector<CUtensorMap> wm((size_t)D.L * 4);
  bool ok = true;
  for (int l = 0; l < D.L; ++l) {
    ok &= map2d(&wm[l * 4 + MK_QKV], wqkv[l], D.d, D.qkvn, kBM);
    ok &= map2d(&wm[l * 4 + MK_WO], wo[l], D.qdim, D.d, kBM);
    ok &= map2d(&wm[l * 4 + MK_GU], wgu[l], D.d, 2 * D.F, kBM);
    ok &= map2d(&wm[l * 4 + MK_DN], wd[l], D.F, D.d, kBM);
  }
  CUtensorMap kvm;
  {
    cuuint64_t dims[3] = {(cuuint64_t)kHD, (cuuint64_t)D.max_len, (cuuint64_t)D.L * 2 * D.maxB * D.Hkv};
    cuuint64_t strides[2] = {(cuuint64_t)kHD * 2, (cuuint64_t)D.max_len * kHD * 2};
    cuuint32_t box[3] = {64, kTP, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    ok &= encode_fn()(&kvm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kv, dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  if (!ok) {
    if (err) *err = "cuTensorMapEncodeTiled failed (persistent kernel maps)";
    return false;
  }
  // segments per tile of each GEMM phase (independent of the batch)
  const int MT = max_tiles(D);
  const int TT[4] = {D.qkvn / kBM, D.d / kBM, 2 * D.F / kBM, D.d / kBM};
  const int KBs[4] = {D.d / kBK, D.qdim / kBK, D.d / kBK, D.F / kBK};
  std::vector<uint8_t> tn(4 * (size_t)MT, 0);
  for (int ph = 0; ph < 4; ++ph) {
    const std::vector<int> n = streamk_nseg(TT[ph], KBs[ph], D.sms);
    P.segs[ph] = 0;
    for (int t = 0; t < TT[ph]; ++t) {
      tn[(size_t)ph * MT + t] = (uint8_t)n[t];
      P.segs[ph] += n[t];
    }
  }
  std::vector<MkLayer> ly(D.L);
  for (int l = 0; l < D.L; ++l) ly[l] = MkLayer{g1[l], g2[l], a[l], b[l], c[l]};
  cudaError_t e = cudaMemcpyAsync(P.wmap, wm.data(), wm.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(P.kvmap, &kvm, sizeof(kvm), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(P.layers, ly.data(), ly.size() * sizeof(MkLayer), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(P.tnseg, tn.data(), tn.size(), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(P.cnt, 0, P.ncnt * 4, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    if (err) *err = std::string("persistent kernel setup: ") + cudaGetErrorString(e);
    return false;
  }
  P.smem = smem_total();
  if (cudaFuncSetAttribute(k_mk_step, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P.smem) != cudaSuccess) {
    cudaGetLastError();
    return true;  // stays disabled
  }
  P.enabled = true;
  return true;
}

bool mk_batch(MkPlan& P, const Dims& D, const Buffers& Bf, int B, std::string* err) {
  if (!P.enabled) return true;
  P.B = B;
  const int S = D.sms, Mpad = mpad_of(D);
  for (int r = 0; r < 3; ++r) {
    MkRowSet& rs = P.rs[r];
    rs.built = false;
    rs.lo = r == 2 ? B : 0;
    rs.hi = r == 1 ? B : 2 * B;
    const int M = rs.hi - rs.lo;
    rs.N = (M + 15) / 16 * 16;
    if (rs.N > kMaxN) continue;
    std::vector<std::vector<MkTask>> lists(S);
    for (int l = 0; l < D.L; ++l) {
      add_norm_phase(lists, l, 0, rs.lo, rs.hi, S);
      add_gemm_phase(lists, l, MK_QKV, D.qkvn / kBM, D.d / kBK, S);
      add_attn_phase(lists, l, B, D.Hkv, S);
      add_gemm_phase(lists, l, MK_WO, D.d / kBM, D.qdim / kBK, S);
      add_norm_phase(lists, l, 1, rs.lo, rs.hi, S);
      add_gemm_phase(lists, l, MK_GU, 2 * D.F / kBM, D.d / kBK, S);
      add_gemm_phase(lists, l, MK_DN, D.d / kBM, D.F / kBK, S);
    }
    size_t mx = 0;
    for (auto& v : lists) mx = std::max(mx, v.size());
    if ((int)mx > rs.maxT) {
      if (err) *err = "persistent kernel: task list longer than its bound";
      return false;
    }
    std::vector<MkTask> flat((size_t)S * rs.maxT);
    std::vector<int> cnts(S);
    for (int c = 0; c < S; ++c) {
      cnts[c] = (int)lists[c].size();
      std::copy(lists[c].begin(), lists[c].end(), flat.begin() + (size_t)c * rs.maxT);
    }
    CUtensorMap xm[3];
    bool ok = map2d(&xm[0], Bf.u, D.d, Mpad, rs.N);
    ok &= map2d(&xm[1], Bf.o, D.qdim, Mpad, rs.N);
    ok &= map2d(&xm[2], Bf.z, D.F, Mpad, rs.N);
    if (!ok) {
      if (err) *err = "cuTensorMapEncodeTiled failed (activation maps)";
      return false;
    }
    cudaError_t e = cudaMemcpy(rs.tasks, flat.data(), flat.size() * sizeof(MkTask), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(rs.ntasks, cnts.data(), cnts.size() * sizeof(int), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(rs.xmap, xm, sizeof(xm), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
      if (err) *err = std::string("persistent kernel task upload: ") + cudaGetErrorString(e);
      return false;
    }
    rs.built = true;
  }
  return true;
}

size_t mk_attn_partial_floats(const Dims& D) {
  return (size_t)std::min(D.maxB, 16) * D.Hkv * kMaxAttnSeg * kApart;
}

bool mk_can_run(const MkPlan& P, const Rows& R) {
  if (!P.enabled || R.B != P.B) return false;
  const int r = (R.lo == 0 && R.hi == 2 * R.B) ? 0 : (R.lo == 0 && R.hi == R.B) ? 1 : (R.lo == R.B) ? 2 : -1;
  return r >= 0 && P.rs[r].built;
}

void mk_launch(const MkPlan& P, const Dims& D, const Buffers& Bf, void* kv, const Rows& R, int save, int saved,
               cudaStream_t s) {
  const int r = (R.lo == 0 && R.hi == 2 * R.B) ? 0 : (R.lo == 0 && R.hi == R.B) ? 1 : 2;
  const MkRowSet& rs = P.rs[r];
  MkParams p{};
  p.tasks = rs.tasks;
  p.ntasks = rs.ntasks;
  p.maxT = rs.maxT;
  p.wmap = P.wmap;
  p.xmap = rs.xmap;
  p.kvmap = P.kvmap;
  p.layers = P.layers;
  p.h = Bf.h;
  p.u = static_cast<__nv_bfloat16*>(Bf.u);
  p.qatt = Bf.qatt;
  p.o = static_cast<__nv_bfloat16*>(Bf.o);
  p.z = static_cast<__nv_bfloat16*>(Bf.z);
  p.kv = static_cast<__nv_bfloat16*>(kv);
  p.rope = Bf.rope;
  p.ctrl = Bf.ctrl;
  p.cnt = P.cnt;
  p.ncnt = P.ncnt;
  p.gpart = P.gpart;
  p.gregion = P.gregion;
  p.apart = P.apart;
  p.q1s = Bf.q1s;
  p.z1s = Bf.z1s;
  p.y1s = Bf.y1s;
  p.cl = CntLayout{D.L, P.max_tiles, D.Hkv, D.maxB};
  p.d = D.d;
  p.qdim = D.qdim;
  p.kvdim = D.kvdim;
  p.F = D.F;
  p.Hq = D.Hq;
  p.Hkv = D.Hkv;
  p.G = D.G;
  p.maxB = D.maxB;
  p.max_len = D.max_len;
  p.B = R.B;
  p.lo = rs.lo;
  p.hi = rs.hi;
  p.N = rs.N;
  p.save = save;
  p.saved = saved;
  p.tnseg = P.tnseg;
  p.segs_wo = P.segs[MK_WO];
  p.segs_dn = P.segs[MK_DN];
  p.eps = D.eps;
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(P.sms);
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = P.smem;
  lc.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;  // every CTA must be resident: they wait on one another
  at[0].val.cooperative = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  cudaLaunchKernelEx(&lc, k_mk_step, p);
}

}  // namespace df
