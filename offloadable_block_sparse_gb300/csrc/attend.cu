// a6 attend: split-K flash-decode over the selected blocks (NOSA explainer
// eq. 8: attention of q over K[selected], V[selected]; NOSA-1B blog,
// sparse_forward: attention over the top-k block indices only).
//
// grid (attend_chunks, U), 128 threads.  CTA (chunk, u) owns every
// attend_chunks-th entry of unit u's selection (blocks still on the host first).  One elected
// thread streams each 32 KiB block (K and V, two 16 KiB boxes with the 128-byte
// swizzle) from the block cache into a 3-stage shared-memory ring with TMA
// (cp.async.bulk.tensor) and an mbarrier per stage.  Warp w handles tokens
// [16w, 16w+16) of every block on the tensor cores (mma.sync m16n8k16, bf16 in,
// fp32 accumulate):
//   S^T (16 tokens x 8 heads) = K (ldmatrix) . q^T           (8 MMAs)
//   online softmax per head in registers (exp2, warp shuffles)
//   P^T fragments by movmatrix.trans of the bf16-packed S^T fragments
//   O^T (128 dims x 8 heads) += V^T (ldmatrix.trans) . P^T   (8 MMAs)
// The four warps' (m, l, O) are merged in shared memory into one partial per
// CTA; the last CTA of the unit (atomic ticket) merges the partials and writes
// the bf16 output.
#include <cooperative_groups.h>

#include "nosa_internal.cuh"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace nosa {

constexpr int kStageBytes = kBlockBytes;            // 32 KiB: [d half][K,V][64 tokens][64 dims]
static_assert(4 * kMaxGroup * kHeadDim * 4 <= 3 * kStageBytes, "warp partials alias the stages");
constexpr int kDeepStages = 6;  // when a unit's CTAs get an SM each
constexpr long long kWaitLimit = kWaitCycles;  // bound of the drain waits after a timeout

__device__ __forceinline__ uint32_t swz(uint32_t stage, int dhalf, int kv, int token, int chunk) {
  return stage + dhalf * 16384 + kv * 8192 + token * 128 + (((chunk ^ (token & 7)) & 7) << 4);
}

// How a unit's split-K partials are merged:
//   kMerge == kMergeTicket : through global scratch; the last CTA of the unit (atomic ticket) merges;
//   kMerge == kMergeCluster: the unit's CTAs form one cluster and merge through distributed shared memory;
//   kMerge == kMergeKernel : CTAs write their partials and exit; attend_merge_kernel merges.
constexpr int kMergeTicket = 0, kMergeCluster = 1, kMergeKernel = 2;

template <int kMerge, int kStages>
__global__ void __launch_bounds__(kAttendThreads, 1)
    attend_kernel(const __grid_constant__ CUtensorMap tmap, LayerState s, const uint16_t* __restrict__ q,
                  uint16_t* __restrict__ out, int fused_fetch) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[kStages];
  __shared__ float wm[4][kMaxGroup], wl[4][kMaxGroup];
  __shared__ int s_blk[kMaxBlocksPerCta], s_slot[kMaxBlocksPerCta], s_new[kMaxBlocksPerCta];
  __shared__ int last, bad_any;
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // [4 warps][8 heads][128] warp partials, aliasing the stages once every copy has landed
  float* wo = reinterpret_cast<float*>(smem);

  const int chunk = blockIdx.x, u = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gr = lane >> 2, t4 = lane & 3;
  const int G = s.G;
  // independent loads first: q fragments, the context length, the unit's selection size
  // q^T as the B operand: b0 = q[head gr][16ks + 2t4 .. +1], b1 = the same +8
  uint32_t qb[8][2];
  {
    const uint16_t* qh = q + ((size_t)u * G + min(gr, G - 1)) * kHeadDim;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qb[ks][0] = gr < G ? *reinterpret_cast<const uint32_t*>(qh + 16 * ks + 2 * t4) : 0u;
      qb[ks][1] = gr < G ? *reinterpret_cast<const uint32_t*>(qh + 16 * ks + 2 * t4 + 8) : 0u;
    }
  }
  const Geometry geo = geometry(*s.T, s.nw, s.sink);  // written two kernels back (append)
  pdl_wait();               // the selection (previous kernel) is needed from here
  pdl_launch_dependents();  // the next layer's append may start
  const int nsel = s.n_sel[u];
  const uint32_t sbase = smem_u32(smem);
  // Work split: the unit's selected blocks are dealt round-robin to its CTAs in an
  // order that puts the blocks still to be copied from the host first, so those
  // few spread one per CTA and their copies start before anything else.
  const int CS = gridDim.x;
  const int nblk = chunk < nsel ? (nsel - chunk + CS - 1) / CS : 0;
  if (warp == 0) {
    // one round trip: every entry's block, slot and fetched mark, requested with the count
    int ev[kMaxCacheSlots / 32][3];
#pragma unroll
    for (int it = 0; it < kMaxCacheSlots / 32; ++it) {
      const int e = it * 32 + lane;
      const bool in = e < s.cap;
      const size_t o = (size_t)u * s.cap + (in ? e : 0);
      ev[it][0] = in ? s.sel[o] : -1;
      ev[it][1] = in ? s.sel_slot[o] : 0;
      ev[it][2] = (in && fused_fetch) ? s.sel_new[o] : 0;
    }
    int n_new = 0;
#pragma unroll
    for (int it = 0; it < kMaxCacheSlots / 32; ++it) {
      const int e = it * 32 + lane;
      n_new += __popc(__ballot_sync(0xffffffffu, e < nsel && ev[it][2]));
    }
    int seen_new = 0, seen_old = 0;
#pragma unroll
    for (int it = 0; it < kMaxCacheSlots / 32; ++it) {
      const int e = it * 32 + lane;
      const bool in = e < nsel;
      const bool nw = in && ev[it][2];
      const unsigned int bn = __ballot_sync(0xffffffffu, nw), bo = __ballot_sync(0xffffffffu, in && !nw);
      const unsigned int below = (1u << lane) - 1u;
      const int pos = nw ? seen_new + __popc(bn & below) : n_new + seen_old + __popc(bo & below);
      seen_new += __popc(bn);
      seen_old += __popc(bo);
      if (in && pos % CS == chunk) {
        const int i = pos / CS;
        int slot = ev[it][1];
        if (slot < 0 || slot >= s.cap) {
          atomicOr(s.err, kErrBounds);
          slot = 0;  // keep the copy in bounds; the result is flagged as invalid
        }
        s_blk[i] = ev[it][0];
        s_slot[i] = slot;
        s_new[i] = nw ? 1 : 0;
      }
    }
  }
  if (tid == 0) {
    prefetch_tmap(&tmap);
    for (int i = 0; i < kStages; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    bad_any = 0;
  }
  __syncthreads();

  // Pipeline.  Blocks without a cache slot (first in this CTA's list) are copied
  // straight from the pinned host store by cp.async of all threads into
  // dedicated stages right away (rows past the context zero-filled) and consumed
  // last, so the host-link latency overlaps the cached blocks.  Cached blocks
  // stream through the remaining stages as a ring, each loaded by one TMA
  // (thread 0) completing on the stage's mbarrier.  Host blocks beyond the
  // dedicated stages (rare) pass through the ring as well.
  int nnew = 0;
  while (nnew < nblk && s_new[nnew]) ++nnew;
  const int ded = min(nnew, kStages - 1);  // dedicated stages 0 .. ded-1
  const int ring = kStages - ded;          // ring stages ded .. kStages-1
  const int nr = nblk - ded;               // ring entries: local entries ded .. nblk-1
  auto host_copy = [&](int e, int st) {    // all threads
    const int rows = (s_blk[e] == geo.nb - 1) ? geo.valid_tail : kBlock;
    const uint16_t* src = s.host_kv + ((size_t)u * s.nb_max + s_blk[e]) * 2 * kBlockElems;
#pragma unroll 4
    for (int j = 0; j < kStageBytes / 16 / kAttendThreads; ++j) {
      const int idx = tid + j * kAttendThreads;  // 16-byte chunk: K|V, row, chunk of the 256-byte row
      const int kv = idx >> 10, r = (idx >> 4) & 63, cc = idx & 15;
      cp_async_16(swz(sbase + st * kStageBytes, cc >> 3, kv, r, cc & 7),
                  src + (size_t)kv * kBlockElems + r * kHeadDim + cc * 8, r < rows ? 16u : 0u);
    }
    cp_async_commit();
  };
  auto issue_ring = [&](int p) {  // ring entry p into stage ded + p % ring
    if (p >= nr) return;
    const int st = ded + p % ring, e = ded + p;
    if (s_new[e]) {
      if (tid == 0) mbar_arrive(&bars[st]);
      host_copy(e, st);
    } else if (tid == 0) {
      const int flat = (s.unit_base + u) * s.cap + s_slot[e];
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&bars[st], kStageBytes);
      tma_load_4d(sbase + st * kStageBytes, &tmap, 0, 0, 0, flat, &bars[st]);
      tma_load_4d(sbase + st * kStageBytes + 16384, &tmap, 64, 0, 0, flat, &bars[st]);
    }
  };
  for (int d = 0; d < ded; ++d) host_copy(d, d);
  for (int p = 0; p < ring; ++p) issue_ring(p);
  int issued = ring;

  const float sl2 = s.scale * 1.4426950408889634f;  // softmax in base 2
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

  const int tok0 = warp * 16;
  // ldmatrix row addresses of this lane (token, 16-byte chunk) before swizzling
  const int tk_k = tok0 + (lane & 7) + (((lane >> 3) & 1) << 3);  // K: matrices (rows 0-7|8-15) x (k lo|hi)
  const int ch_k = lane >> 4;
  const int tk_v = tok0 + (lane & 7) + ((lane >> 4) << 3);        // V^T: (d lo|hi) x (tokens 0-7|8-15)
  const int ch_v = (lane >> 3) & 1;

  // one 64-token block in stage memory stg: warp's 16 tokens, online softmax, PV; fetched
  // blocks are also written to their cache slot for later steps
  auto process = [&](uint32_t stg, int e) {
    const int valid = (s_blk[e] == geo.nb - 1) ? geo.valid_tail : kBlock;
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
      if (tok0 + gr >= valid) acc[0] = acc[1] = -INFINITY;
      if (tok0 + gr + 8 >= valid) acc[2] = acc[3] = -INFINITY;
      float mx0 = fmaxf(acc[0], acc[2]), mx1 = fmaxf(acc[1], acc[3]);
#pragma unroll
      for (int o2 = 4; o2 < 32; o2 <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);  // finite: token tok0 is valid
      const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
      const float p0 = exp2f(acc[0] - mn0), p1 = exp2f(acc[1] - mn1);
      const float p2 = exp2f(acc[2] - mn0), p3 = exp2f(acc[3] - mn1);
      l0 = l0 * al0 + p0 + p2;
      l1 = l1 * al1 + p1 + p3;
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][0] *= al0;
        o[mt][1] *= al1;
        o[mt][2] *= al0;
        o[mt][3] *= al1;
      }
      const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p0, p1));  // tokens 0-7 of the tile
      const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p2, p3));  // tokens 8-15
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int dch = 2 * mt + ch_v;
        uint32_t a[4];
        ldsm_x4_trans(a, swz(stg, dch >> 3, 1, tk_v, dch & 7));
        mma_16816(o[mt], a, pb0, pb1);
      }
    }
    if (s_new[e]) {
      uint16_t* dst = s.cache + ((size_t)u * s.cap + s_slot[e]) * 2 * kBlockElems;
#pragma unroll 4
      for (int j = 0; j < kStageBytes / 16 / kAttendThreads; ++j) {
        const int idx = tid + j * kAttendThreads;
        const int kv = idx >> 10, r = (idx >> 4) & 63, cc = idx & 15;
        uint4 v;
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "r"(swz(stg, cc >> 3, kv, r, cc & 7)));
        *reinterpret_cast<uint4*>(dst + (size_t)kv * kBlockElems + r * kHeadDim + cc * 8) = v;
      }
    }
  };

  int consumed = 0;
  for (int p = 0; p < nr; ++p) {
    const int st = ded + p % ring, e = ded + p;
    // a negative limit (a test hook) gives up without waiting, so the timeout path runs every time
    const bool okw = s.wait_limit >= 0 && mbar_wait_bounded(&bars[st], (uint32_t)((p / ring) & 1), s.wait_limit);
    if (s_new[e]) cp_async_wait_all();  // a host block that passed through the ring
    if (__syncthreads_or(!okw)) {
      if (tid == 0) atomicOr(s.err, kErrTimeout);
      bad_any = 1;
      break;
    }
    consumed = p + 1;
    process(sbase + st * kStageBytes, e);
    __syncthreads();  // every warp is done with this stage
    issue_ring(issued);
    ++issued;
  }
  cp_async_wait_all();
  __syncthreads();  // the dedicated host blocks have landed
  if (!bad_any)
    for (int d = 0; d < ded; ++d) process(sbase + d * kStageBytes, d);
  if (bad_any && tid == 0) {  // drain copies still in flight before the shared memory is reused
    for (int p = consumed; p < min(issued, nr); ++p)
      mbar_wait_bounded(&bars[ded + p % ring], (uint32_t)((p / ring) & 1), kWaitLimit);
  }
  __syncthreads();
  // warp partials -> shared memory
#pragma unroll
  for (int o2 = 4; o2 < 32; o2 <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o2);
  }
  if (gr == 0) {
    wm[warp][2 * t4] = m0;
    wm[warp][2 * t4 + 1] = m1;
    wl[warp][2 * t4] = l0;
    wl[warp][2 * t4 + 1] = l1;
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    float* w0 = wo + ((warp * kMaxGroup + 2 * t4) * kHeadDim);
    float* w1 = wo + ((warp * kMaxGroup + 2 * t4 + 1) * kHeadDim);
    w0[16 * mt + gr] = o[mt][0];
    w1[16 * mt + gr] = o[mt][1];
    w0[16 * mt + gr + 8] = o[mt][2];
    w1[16 * mt + gr + 8] = o[mt][3];
  }
  __syncthreads();
  // CTA partial (base-2 max, sum, unnormalised output) for each head
  const int x = tid;  // head dimension
  __shared__ float cp_m[kMaxGroup], cp_l[kMaxGroup], cp_o[kMaxGroup][kHeadDim];
  float* part0 = s.apart + ((size_t)u * s.attend_chunks + chunk) * kMaxGroup * kPartStride;
  for (int h = 0; h < G; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, wm[w][h]);
    float L = 0.f, O = 0.f;
    if (M > -INFINITY) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float f = exp2f(wm[w][h] - M);
        L += wl[w][h] * f;
        O += wo[(w * kMaxGroup + h) * kHeadDim + x] * f;
      }
    }
    if constexpr (kMerge == kMergeCluster) {
      if (x == 0) {
        cp_m[h] = M;
        cp_l[h] = L;
      }
      cp_o[h][x] = O;
    } else {
      float* part = part0 + h * kPartStride;
      if (x == 0) {
        part[0] = M;
        part[1] = L;
      }
      part[2 + x] = O;
    }
  }
  if constexpr (kMerge == kMergeKernel) return;
  if constexpr (kMerge == kMergeCluster) {
    // every CTA of the unit merges the heads h = rank, rank + CS, ... from all CTAs' partials
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank(), CS = (int)cluster.num_blocks();
    cluster.sync();
    for (int h = rank; h < G; h += CS) {
      float mr[16], M = -INFINITY;
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        mr[r] = r < CS ? *cluster.map_shared_rank(&cp_m[h], r) : -INFINITY;
        M = fmaxf(M, mr[r]);
      }
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        if (r < CS && mr[r] > -INFINITY) {
          const float f = exp2f(mr[r] - M);
          L += *cluster.map_shared_rank(&cp_l[h], r) * f;
          O += *cluster.map_shared_rank(&cp_o[h][x], r) * f;
        }
      }
      const float res = L > 0.f ? O / L : 0.f;
      out[((size_t)u * G + h) * kHeadDim + x] = __bfloat16_as_ushort(__float2bfloat16_rn(res));
    }
    cluster.sync();  // keep every CTA's partial alive until all remote reads are done
    return;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned int t = atomicAdd(&s.tickets[s.U + u], 1u);
    last = (t == (unsigned int)s.attend_chunks - 1);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (tid == 0) s.tickets[s.U + u] = 0;
  // merge the unit's partials: all (m, l) pairs in one round trip, then every o value in flight at once
  const int nch = s.attend_chunks;
  const float* pu = s.apart + (size_t)u * nch * kMaxGroup * kPartStride;
  float* pm = reinterpret_cast<float*>(smem);        // [nch][8] scale factors
  float* pl = pm + nch * kMaxGroup;                  // [nch][8] sums
  __shared__ float Mh[kMaxGroup], Lh[kMaxGroup];
  for (int idx = tid; idx < nch * G; idx += blockDim.x) {
    const int j = idx / G, h = idx % G;
    const float* p = pu + ((size_t)j * kMaxGroup + h) * kPartStride;
    pm[j * kMaxGroup + h] = __ldcg(p);
    pl[j * kMaxGroup + h] = __ldcg(p + 1);
  }
  __syncthreads();
  if (tid < G) {
    float M = -INFINITY;
    for (int j = 0; j < nch; ++j) M = fmaxf(M, pm[j * kMaxGroup + tid]);
    float L = 0.f;
    for (int j = 0; j < nch; ++j) {
      const float mj = pm[j * kMaxGroup + tid];
      const float f = (mj > -INFINITY) ? exp2f(mj - M) : 0.f;
      pm[j * kMaxGroup + tid] = f;
      L += pl[j * kMaxGroup + tid] * f;
    }
    Mh[tid] = M;
    Lh[tid] = L;
  }
  __syncthreads();
  // o partials: 8 chunks x 8 heads of loads in flight per batch
  float O[kMaxGroup];
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h) O[h] = 0.f;
  for (int j0 = 0; j0 < nch; j0 += 8) {
    float ov[8][kMaxGroup];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int h = 0; h < kMaxGroup; ++h)
        ov[r][h] = (j0 + r < nch && h < G) ? __ldcg(pu + ((size_t)(j0 + r) * kMaxGroup + h) * kPartStride + 2 + x)
                                           : 0.f;
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int h = 0; h < kMaxGroup; ++h)
        if (j0 + r < nch && h < G) O[h] = fmaf(ov[r][h], pm[(j0 + r) * kMaxGroup + h], O[h]);
  }
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h) {
    if (h >= G) break;
    const float r = Lh[h] > 0.f ? O[h] / Lh[h] : 0.f;
    out[((size_t)u * G + h) * kHeadDim + x] = __bfloat16_as_ushort(__float2bfloat16_rn(r));
  }
}

size_t attend_smem_bytes(int stages) { return 1024 + (size_t)stages * kStageBytes; }

// Merges the split-K partials of one (head, unit): grid (group, U), 128 threads
// (one per head dimension).  Launched as a programmatic dependent of the
// attention kernel; every (m, l) pair and o value is requested at once.
__global__ void __launch_bounds__(kHeadDim) attend_merge_kernel(LayerState s, uint16_t* __restrict__ out) {
  __shared__ float fm[256], fl[256];
  pdl_wait();  // the partials are written by the previous kernel
  pdl_launch_dependents();
  const int h = blockIdx.x, u = blockIdx.y, x = threadIdx.x;
  const int nch = s.attend_chunks;
  const float* pb = s.apart + ((size_t)u * nch * kMaxGroup + h) * kPartStride;
  for (int j = x; j < nch; j += blockDim.x) {
    fm[j] = pb[(size_t)j * kMaxGroup * kPartStride];
    fl[j] = pb[(size_t)j * kMaxGroup * kPartStride + 1];
  }
  float ov[16];
  const int first = min(nch, 16);
#pragma unroll
  for (int j = 0; j < 16; ++j) ov[j] = j < first ? pb[(size_t)j * kMaxGroup * kPartStride + 2 + x] : 0.f;
  __syncthreads();
  float M = -INFINITY;
  for (int j = 0; j < nch; ++j) M = fmaxf(M, fm[j]);
  float L = 0.f, O = 0.f;
  if (M > -INFINITY) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < first && fm[j] > -INFINITY) {
        const float f = exp2f(fm[j] - M);
        L += fl[j] * f;
        O = fmaf(ov[j], f, O);
      }
    for (int j = 16; j < nch; ++j)
      if (fm[j] > -INFINITY) {
        const float f = exp2f(fm[j] - M);
        L += fl[j] * f;
        O = fmaf(pb[(size_t)j * kMaxGroup * kPartStride + 2 + x], f, O);
      }
  }
  const float r = L > 0.f ? O / L : 0.f;
  out[((size_t)u * s.G + h) * kHeadDim + x] = __bfloat16_as_ushort(__float2bfloat16_rn(r));
}

template <int M, int S>
static cudaError_t set_attend_attrs() {
  cudaError_t e = cudaFuncSetAttribute(attend_kernel<M, S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)attend_smem_bytes(S));
  if (e != cudaSuccess || M != kMergeCluster) return e;
  return cudaFuncSetAttribute(attend_kernel<M, S>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

cudaError_t init_attend() {
  cudaError_t e = set_attend_attrs<kMergeTicket, kAttendStages>();
  if (e == cudaSuccess) e = set_attend_attrs<kMergeCluster, kAttendStages>();
  if (e == cudaSuccess) e = set_attend_attrs<kMergeCluster, kDeepStages>();
  if (e == cudaSuccess) e = set_attend_attrs<kMergeKernel, kAttendStages>();
  if (e == cudaSuccess) e = set_attend_attrs<kMergeKernel, kDeepStages>();
  return e;
}

template <int M, int S>
static cudaError_t launch_attend_t(const LayerState& s, const CUtensorMap* tmap, const uint16_t* q, uint16_t* out,
                                   int fused_fetch, bool pdl, cudaStream_t st) {
  return launch_ex(attend_kernel<M, S>, dim3(s.attend_chunks, s.U), dim3(kAttendThreads), attend_smem_bytes(S), st,
                   pdl, M == kMergeCluster ? s.attend_chunks : 0, *tmap, s, q, out, fused_fetch);
}

cudaError_t launch_attend(const LayerState& s, const CUtensorMap* tmap, const uint16_t* q, uint16_t* out,
                          int fused_fetch, bool pdl, cudaStream_t st) {
  if (s.attend_mode == kMergeKernel) {
    cudaError_t e = s.attend_deep ? launch_attend_t<kMergeKernel, kDeepStages>(s, tmap, q, out, fused_fetch, pdl, st)
                                  : launch_attend_t<kMergeKernel, kAttendStages>(s, tmap, q, out, fused_fetch, pdl, st);
    if (e != cudaSuccess) return e;
    return launch_ex(attend_merge_kernel, dim3(s.G, s.U), dim3(kHeadDim), 0, st, true, 0, s, out);
  }
  if (s.attend_mode == kMergeTicket)
    return launch_attend_t<kMergeTicket, kAttendStages>(s, tmap, q, out, fused_fetch, pdl, st);
  if (s.attend_deep) return launch_attend_t<kMergeCluster, kDeepStages>(s, tmap, q, out, fused_fetch, pdl, st);
  return launch_attend_t<kMergeCluster, kAttendStages>(s, tmap, q, out, fused_fetch, pdl, st);
}

// Largest cluster of attend CTAs (with this kernel's shared memory) the device can schedule.
int attend_max_cluster(bool deep) {
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kAttendThreads);
  cfg.dynamicSmemBytes = attend_smem_bytes(deep ? kDeepStages : kAttendStages);
  int best = 1;
  for (int c : {8, 4, 2}) {
    cfg.gridDim = dim3(c, 1);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t e =
        deep ? cudaOccupancyMaxActiveClusters(&n, attend_kernel<kMergeCluster, kDeepStages>, &cfg)
             : cudaOccupancyMaxActiveClusters(&n, attend_kernel<kMergeCluster, kAttendStages>, &cfg);
    if (e == cudaSuccess && n > 0) {
      best = c;
      break;
    }
    (void)cudaGetLastError();
  }
  return best;
}

}  // namespace nosa
