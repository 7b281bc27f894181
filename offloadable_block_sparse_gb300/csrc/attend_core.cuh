// Split-K flash-decode core shared by the attention kernel and the fused decode
// kernel (NOSA explainer eq. 8: attention of q over K[selected], V[selected]).
//
// A "worker" is a team of four warps (128 threads) that owns a list of selected
// blocks of one unit.  Blocks without a cache slot come first in the list; they
// are copied straight from the pinned host store by cp.async of all the team's
// threads into dedicated stages (rows past the context zero-filled) and are
// consumed last, so the host-link latency overlaps the cached blocks.  Cached
// blocks stream through the remaining stages as a ring, each 32 KiB block (K and
// V, two 16 KiB boxes with the 128-byte swizzle) loaded by one TMA
// (cp.async.bulk.tensor) issued by the team's first thread and completing on the
// stage's mbarrier.  Warp w of the team handles tokens [16w, 16w+16) of every
// block on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate):
//   S^T (16 tokens x 8 heads) = K (ldmatrix) . q^T           (8 MMAs)
//   online softmax per head in registers (exp2, warp shuffles)
//   P^T fragments by movmatrix.trans of the bf16-packed S^T fragments
//   O^T (128 dims x 8 heads) += V^T (ldmatrix.trans) . P^T   (8 MMAs)
// Blocks copied from the host are also written to their cache slot for later steps.
#pragma once

#include "nosa_internal.cuh"
#include "ptx.cuh"

namespace nosa {

constexpr int kStageBytes = kBlockBytes;  // 32 KiB: [d half][K,V][64 tokens][64 dims]
constexpr int kTeamThreads = 128;

__device__ __forceinline__ uint32_t swz(uint32_t stage, int dhalf, int kv, int token, int chunk) {
  return stage + dhalf * 16384 + kv * 8192 + token * 128 + (((chunk ^ (token & 7)) & 7) << 4);
}

// A named barrier over the 128 threads of one team (id 0 with a 128-thread CTA is __syncthreads).
struct Team {
  uint32_t id;
  __device__ __forceinline__ void sync() const {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(kTeamThreads) : "memory");
  }
  __device__ __forceinline__ bool sync_or(bool p) const {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n bar.red.or.pred po, %2, %3, pi;\n"
        " selp.u32 %0, 1, 0, po;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)p), "r"(id), "r"(kTeamThreads)
        : "memory");
    return r != 0;
  }
};

// q^T as the B operand of the score MMA: b0 = q[head gr][16ks + 2t4 .. +1], b1 = the same +8.
__device__ __forceinline__ void load_q_frags(uint32_t (&qb)[8][2], const uint16_t* q, int u, int G, int lane) {
  const int gr = lane >> 2, t4 = lane & 3;
  const uint16_t* qh = q + ((size_t)u * G + min(gr, G - 1)) * kHeadDim;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    qb[ks][0] = gr < G ? *reinterpret_cast<const uint32_t*>(qh + 16 * ks + 2 * t4) : 0u;
    qb[ks][1] = gr < G ? *reinterpret_cast<const uint32_t*>(qh + 16 * ks + 2 * t4 + 8) : 0u;
  }
}

// Copies block `blk` of unit u from the pinned host store into the stage at `stage`
// (K then V, with the attention's swizzle; rows past the context zero-filled) by
// cp.async of the team's 128 threads, as one commit group per thread.
__device__ __forceinline__ void host_block_copy(const LayerState& s, const Geometry& geo, int u, int blk,
                                                uint32_t stage, int ttid) {
  const int rows = (blk == geo.nb - 1) ? geo.valid_tail : kBlock;
  const uint16_t* src = s.host_kv + ((size_t)u * s.nb_max + blk) * 2 * kBlockElems;
#pragma unroll 4
  for (int j = 0; j < kStageBytes / 16 / kTeamThreads; ++j) {
    const int idx = ttid + j * kTeamThreads;  // 16-byte chunk: K|V, row, chunk of the 256-byte row
    const int kv = idx >> 10, r = (idx >> 4) & 63, cc = idx & 15;
    cp_async_16(swz(stage, cc >> 3, kv, r, cc & 7), src + (size_t)kv * kBlockElems + r * kHeadDim + cc * 8,
                r < rows ? 16u : 0u);
  }
  cp_async_commit();
}

// One warp's running softmax state: base-2 maxima and sums for heads 2t4, 2t4+1, and
// O^T fragments (8 tiles of 16 dims).
struct WarpAcc {
  float m0, m1, l0, l1;
  float o[8][4];
  __device__ __forceinline__ void init() {
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  }
};

// Runs one worker over its list (blk, slot, isnew; n entries, blocks without a slot
// first) with `nst` stages at sbase and their mbarriers `bars` (initialised, count 1).
// With s.dma_bias, sebuf (nst x 64 floats, 16-byte aligned) receives each staged
// block's per-token eviction scores, added to the logits.  Returns false if a staged-block wait
// gave up: the error word has the timeout bit, copies in flight have been drained, and the
// worker's softmax sums are NaN, so every output its partial reaches is NaN rather than a
// plausible value.  ttid: thread index within the team.
__device__ __forceinline__ bool attend_worker(const CUtensorMap* tmap, const LayerState& s, const Geometry& geo,
                                              int u, const uint32_t (&qb)[8][2], const int* blk, const int* slot,
                                              const int* isnew, int n, uint32_t sbase, uint64_t* bars, int nst,
                                              float* sebuf, Team team, int ttid, WarpAcc& A) {
  const int lane = ttid & 31, warp = ttid >> 5;
  const int gr = lane >> 2, t4 = lane & 3;
  int nnew = 0;
  while (nnew < n && isnew[nnew]) ++nnew;
  const int ded = min(nnew, nst - 1);  // dedicated stages 0 .. ded-1
  const int ring = nst - ded;          // ring stages ded .. nst-1
  const int nr = n - ded;              // ring entries: local entries ded .. n-1
  const bool dma = s.dma_bias != 0;
  // the block's 64 per-token eviction scores (256 bytes, 256-byte aligned rows)
  auto se_src = [&](int e) { return s.se_tok + (size_t)u * s.se_stride + (size_t)kBlock * blk[e]; };
  auto host_copy = [&](int e, int st) {
    host_block_copy(s, geo, u, blk[e], sbase + st * kStageBytes, ttid);
    if (dma) {
      if (ttid < kBlock / 4) cp_async_16(smem_u32(sebuf + st * kBlock) + 16 * ttid, se_src(e) + 4 * ttid, 16);
      cp_async_commit();
    }
  };
  auto issue_ring = [&](int p) {  // ring entry p into stage ded + p % ring
    if (p >= nr) return;
    const int st = ded + p % ring, e = ded + p;
    if (isnew[e]) {
      if (ttid == 0) mbar_arrive(&bars[st]);
      host_copy(e, st);
    } else if (ttid == 0) {
      const int flat = (s.unit_base + u) * s.cslots + slot[e];
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&bars[st], kStageBytes + (dma ? kBlock * 4 : 0));
      tma_load_4d(sbase + st * kStageBytes, tmap, 0, 0, 0, flat, &bars[st]);
      tma_load_4d(sbase + st * kStageBytes + 16384, tmap, 64, 0, 0, flat, &bars[st]);
      if (dma) bulk_copy_g2s(smem_u32(sebuf + st * kBlock), se_src(e), kBlock * 4, &bars[st]);
    }
  };
  for (int d = 0; d < ded; ++d) host_copy(d, d);
  for (int p = 0; p < ring; ++p) issue_ring(p);
  int issued = ring;

  const float sl2 = s.scale * 1.4426950408889634f;  // softmax in base 2
  const int tok0 = warp * 16;
  // ldmatrix row addresses of this lane (token, 16-byte chunk) before swizzling
  const int tk_k = tok0 + (lane & 7) + (((lane >> 3) & 1) << 3);  // K: matrices (rows 0-7|8-15) x (k lo|hi)
  const int ch_k = lane >> 4;
  const int tk_v = tok0 + (lane & 7) + ((lane >> 4) << 3);        // V^T: (d lo|hi) x (tokens 0-7|8-15)
  const int ch_v = (lane >> 3) & 1;

  auto process = [&](int st, int e) {
    const uint32_t stg = sbase + st * kStageBytes;
    const int valid = (blk[e] == geo.nb - 1) ? geo.valid_tail : kBlock;
    if (tok0 < valid) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int dch = 2 * ks + ch_k;
        uint32_t a[4];
        ldsm_x4(a, swz(stg, dch >> 3, 0, tk_k, dch & 7));
        mma_16816(acc, a, qb[ks][0], qb[ks][1]);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[j] *= sl2;
      if (dma) {  // natural-log bias in base-2 units
        const float b0 = sebuf[st * kBlock + tok0 + gr] * 1.4426950408889634f;
        const float b1 = sebuf[st * kBlock + tok0 + gr + 8] * 1.4426950408889634f;
        acc[0] += b0;
        acc[1] += b0;
        acc[2] += b1;
        acc[3] += b1;
      }
      if (tok0 + gr >= valid) acc[0] = acc[1] = -INFINITY;
      if (tok0 + gr + 8 >= valid) acc[2] = acc[3] = -INFINITY;
      float mx0 = fmaxf(acc[0], acc[2]), mx1 = fmaxf(acc[1], acc[3]);
#pragma unroll
      for (int o2 = 4; o2 < 32; o2 <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
      }
      const float mn0 = fmaxf(A.m0, mx0), mn1 = fmaxf(A.m1, mx1);  // finite: token tok0 is valid
      const float al0 = exp2f(A.m0 - mn0), al1 = exp2f(A.m1 - mn1);
      const float p0 = exp2f(acc[0] - mn0), p1 = exp2f(acc[1] - mn1);
      const float p2 = exp2f(acc[2] - mn0), p3 = exp2f(acc[3] - mn1);
      A.l0 = A.l0 * al0 + p0 + p2;
      A.l1 = A.l1 * al1 + p1 + p3;
      A.m0 = mn0;
      A.m1 = mn1;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        A.o[mt][0] *= al0;
        A.o[mt][1] *= al1;
        A.o[mt][2] *= al0;
        A.o[mt][3] *= al1;
      }
      const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p0, p1));  // tokens 0-7 of the tile
      const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p2, p3));  // tokens 8-15
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int dch = 2 * mt + ch_v;
        uint32_t a[4];
        ldsm_x4_trans(a, swz(stg, dch >> 3, 1, tk_v, dch & 7));
        mma_16816(A.o[mt], a, pb0, pb1);
      }
    }
    if (isnew[e]) {
      uint16_t* dst = s.cache + ((size_t)u * s.cslots + slot[e]) * 2 * kBlockElems;
#pragma unroll 4
      for (int j = 0; j < kStageBytes / 16 / kTeamThreads; ++j) {
        const int idx = ttid + j * kTeamThreads;
        const int kv = idx >> 10, r = (idx >> 4) & 63, cc = idx & 15;
        uint4 v;
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "r"(swz(stg, cc >> 3, kv, r, cc & 7)));
        *reinterpret_cast<uint4*>(dst + (size_t)kv * kBlockElems + r * kHeadDim + cc * 8) = v;
      }
    }
  };

  bool bad = false;
  int consumed = 0;
  for (int p = 0; p < nr; ++p) {
    const int st = ded + p % ring, e = ded + p;
    // a negative limit (a test hook) gives up without waiting, so the timeout path runs every time
    const bool okw = s.wait_limit >= 0 && mbar_wait_bounded(&bars[st], (uint32_t)((p / ring) & 1), s.wait_limit);
    if (isnew[e]) cp_async_wait_all();  // a host block that passed through the ring
    if (team.sync_or(!okw)) {
      if (ttid == 0) atomicOr(s.err, kErrTimeout);
      bad = true;
      break;
    }
    consumed = p + 1;
    process(st, e);
    team.sync();  // every warp is done with this stage
    issue_ring(issued);
    ++issued;
  }
  cp_async_wait_all();
  team.sync();  // the dedicated host blocks have landed
  if (!bad)
    for (int d = 0; d < ded; ++d) process(d, d);
  if (bad && ttid == 0) {  // drain copies still in flight before the shared memory is reused
    for (int p = consumed; p < min(issued, nr); ++p)
      mbar_wait_bounded(&bars[ded + p % ring], (uint32_t)((p / ring) & 1), kWaitCycles);
  }
  if (bad) A.l0 = A.l1 = __int_as_float(0x7fc00000);  // NaN: the merged outputs of this unit are NaN
  (void)gr;
  (void)t4;
  return !bad;
}

// Reduces the warps' softmax state to one (m, l, o) per head: warp partials go to
// shared memory (wm, wl [nwarps][8], wo [nwarps][8][128]); one thread per head forms
// the head's maximum, sum and per-warp scale factors (written over wm), then every
// thread of the CTA combines output elements.  Call with every thread of the CTA;
// contains __syncthreads.  emit(h, x, M, L, O) is called once per head h < G and
// dimension x < 128.
template <int kWarps, typename Emit>
__device__ __forceinline__ void cta_partial(const WarpAcc& A, float (*wm)[kMaxGroup], float (*wl)[kMaxGroup],
                                            float* wo, int G, Emit emit) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gr = lane >> 2, t4 = lane & 3;
  float l0 = A.l0, l1 = A.l1;
#pragma unroll
  for (int o2 = 4; o2 < 32; o2 <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o2);
  }
  if (gr == 0) {
    wm[warp][2 * t4] = A.m0;
    wm[warp][2 * t4 + 1] = A.m1;
    wl[warp][2 * t4] = l0;
    wl[warp][2 * t4 + 1] = l1;
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    float* w0 = wo + ((warp * kMaxGroup + 2 * t4) * kHeadDim);
    float* w1 = wo + ((warp * kMaxGroup + 2 * t4 + 1) * kHeadDim);
    w0[16 * mt + gr] = A.o[mt][0];
    w1[16 * mt + gr] = A.o[mt][1];
    w0[16 * mt + gr + 8] = A.o[mt][2];
    w1[16 * mt + gr + 8] = A.o[mt][3];
  }
  __shared__ float head_m[kMaxGroup], head_l[kMaxGroup];
  __syncthreads();
  if (tid < G) {
    const int h = tid;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w][h]);
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = M > -INFINITY ? exp2f(wm[w][h] - M) : 0.f;
      L += wl[w][h] * f;
      wm[w][h] = f;  // the warp's scale factor from here on
    }
    head_m[h] = M;
    head_l[h] = L;
  }
  __syncthreads();
  for (int idx = tid; idx < G * kHeadDim; idx += blockDim.x) {
    const int h = idx >> 7, x = idx & (kHeadDim - 1);
    float O = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) O = fmaf(wo[(w * kMaxGroup + h) * kHeadDim + x], wm[w][h], O);
    emit(h, x, head_m[h], head_l[h], O);
  }
}

}  // namespace nosa
