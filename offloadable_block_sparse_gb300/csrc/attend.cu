// a6 attend: split-K flash-decode over the selected blocks (NOSA explainer
// eq. 8: attention of q over K[selected], V[selected]; NOSA-1B blog,
// sparse_forward: attention over the top-k block indices only).
//
// grid (U, attend_chunks) — (attend_chunks, U) when a unit's CTAs form one cluster —
// 128 threads: one worker of the shared core (a team of four warps, TMA ring over the
// block cache, host blocks by cp.async) per CTA.  CTAs start in the order of their
// linear index, so with chunks along y every unit's chunk 0 (which holds its first block
// still on the host) starts in the first wave, then chunk 1, ...: the host-link copies of
// all units are under way from the start rather than a wave at a time.  CTA (chunk, u) owns every attend_chunks-th entry of unit u's selection
// (blocks still on the host first).  The four warps' (m, l, O) are merged in
// shared memory into one partial per CTA; the unit's partials are then merged
// through the cluster's distributed shared memory, by a merge kernel, or by the
// last CTA of the unit (atomic ticket), which writes the bf16 output.
#include <cooperative_groups.h>

#include "attend_core.cuh"
#include "host.h"

namespace cg = cooperative_groups;

namespace nosa {

static_assert(4 * kMaxGroup * kHeadDim * 4 <= 3 * kStageBytes, "warp partials alias the stages");

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
  __shared__ int last;
  __shared__ __align__(16) float sebuf[kStages][kBlock];  // per-token eviction scores of the staged blocks
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // [4 warps][8 heads][128] warp partials, aliasing the stages once every copy has landed
  float* wo = reinterpret_cast<float*>(smem);

  constexpr bool kChunksAlongX = kMerge == kMergeCluster;
  const int chunk = kChunksAlongX ? blockIdx.x : blockIdx.y, u = kChunksAlongX ? blockIdx.y : blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = s.G;
  // Everything is read after the wait (q, the context length, the selection): the previous
  // kernel may be the append that sets T, or the kernel that wrote q.  These loads and the
  // selection entries below go out together, one round trip.
  pdl_wait();
  pdl_launch_dependents();  // the next layer's append may start
  uint32_t qb[8][2];
  load_q_frags(qb, q, u, G, lane);
  const int T = *s.T;
  const int nsel_in = s.n_sel[u];
  // a count beyond the selection arrays (possible only for a caller-supplied selection) is
  // clamped, so that no list index leaves the arrays, and flagged
  const int nsel = min(max(nsel_in, 0), s.cap);
  if (nsel != nsel_in && tid == 0 && chunk == 0) atomicOr(s.err, kErrBounds);
  const Geometry geo = geometry(T, s.nw, s.sink);
  const uint32_t sbase = smem_u32(smem);
  // Work split: the unit's selected blocks are dealt round-robin to its CTAs in an
  // order that puts the blocks still to be copied from the host first, so those
  // few spread one per CTA.  Each unit starts dealing at its own chunk (u mod CS), so
  // neighbouring units' host blocks land on different chunks and every wave of CTAs
  // carries about the same share of host copies: the link stays busy for the whole
  // launch while the cached blocks stream from HBM, instead of the first waves waiting
  // on the link and the last ones on HBM.
  const int CS = kChunksAlongX ? gridDim.x : gridDim.y;  // the unit's CTAs
  const int c0 = (chunk - u % CS + CS) % CS;             // this CTA's dealing positions: c0, c0 + CS, ...
  const int nblk = c0 < nsel ? (nsel - c0 + CS - 1) / CS : 0;
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
      if (in && pos % CS == c0) {
        const int i = pos / CS;
        int slot = ev[it][1];
        if (slot < 0 || slot >= s.cslots) {
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
  }
  __syncthreads();

  WarpAcc A;
  A.init();
  attend_worker(&tmap, s, geo, u, qb, s_blk, s_slot, s_new, nblk, sbase, bars, kStages, &sebuf[0][0], Team{0}, tid, A);
  __syncthreads();  // every copy has landed (or was drained): the stages can hold the warp partials

  // CTA partial (base-2 max, sum, unnormalised output) for each head
  __shared__ float cp_m[kMaxGroup], cp_l[kMaxGroup], cp_o[kMaxGroup][kHeadDim];
  float* part0 = s.apart + ((size_t)u * s.attend_chunks + chunk) * kMaxGroup * kPartStride;
  cta_partial<4>(A, wm, wl, wo, G, [&](int h, int x, float M, float L, float O) {
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
  });
  const int x = tid;  // head dimension
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

cudaError_t launch_attend_merge(const LayerState& s, uint16_t* out, cudaStream_t st) {
  return launch_ex(attend_merge_kernel, dim3(s.G, s.U), dim3(kHeadDim), 0, st, true, 0, s, out);
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
  if (e == cudaSuccess) e = set_attend_attrs<kMergeKernel, kAttendStages>();
  return e;
}

template <int M, int S>
static cudaError_t launch_attend_t(const LayerState& s, const CUtensorMap* tmap, const uint16_t* q, uint16_t* out,
                                   int fused_fetch, bool pdl, cudaStream_t st) {
  const dim3 grid = M == kMergeCluster ? dim3(s.attend_chunks, s.U) : dim3(s.U, s.attend_chunks);
  return launch_ex(attend_kernel<M, S>, grid, dim3(kAttendThreads), attend_smem_bytes(S), st, pdl,
                   M == kMergeCluster ? s.attend_chunks : 0, *tmap, s, q, out, fused_fetch);
}

cudaError_t launch_attend(const LayerState& s, const CUtensorMap* tmap, const uint16_t* q, uint16_t* out,
                          int fused_fetch, bool pdl, cudaStream_t st) {
  if (s.attend_mode == kMergeKernel) {
    cudaError_t e = launch_attend_t<kMergeKernel, kAttendStages>(s, tmap, q, out, fused_fetch, pdl, st);
    if (e != cudaSuccess) return e;
    return launch_attend_merge(s, out, st);
  }
  if (s.attend_mode == kMergeTicket)
    return launch_attend_t<kMergeTicket, kAttendStages>(s, tmap, q, out, fused_fetch, pdl, st);
  return launch_attend_t<kMergeCluster, kAttendStages>(s, tmap, q, out, fused_fetch, pdl, st);
}

// Largest cluster of attend CTAs (with this kernel's shared memory) the device can schedule.
int attend_max_cluster() {
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kAttendThreads);
  cfg.dynamicSmemBytes = attend_smem_bytes(kAttendStages);
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
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, attend_kernel<kMergeCluster, kAttendStages>, &cfg);
    if (e == cudaSuccess && n > 0) {
      best = c;
      break;
    }
    (void)cudaGetLastError();
  }
  return best;
}

}  // namespace nosa
