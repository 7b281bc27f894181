// NOSA_S sparse prefill: a prompt appended to an empty layer, every prompt position
// attended over its own block selection (NOSA wiki, "Results": NOSA_S is sparse in
// prefill as well as in decoding; NOSA wiki, "How NOSA works": the query-agnostic
// part never re-selects a block it dropped at an earlier step).  The selection for
// position t is the decode step's selection at T = t + 1 with the eviction state
// carried from position t - 1, so the positions are selected in order, and their
// attention then runs in one launch.
//
//   1. bulk append (append.cu): host store, eviction scores, compressed keys.
//   2. prefill_select_kernel: one CTA per unit walks the positions.  Positions are
//      scored P at a time (one load of every compressed-key tile for P queries); each
//      position then runs the two-part selector of the decode step (select_core.cuh)
//      with the geometry of T = t + 1: query-aware scores over the windows complete
//      at T, pooled eviction scores of the blocks whose windows are complete at T
//      (only the last two blocks can differ from the whole prompt's), the sticky
//      eviction update and the slot pairing.  The selection is written to the
//      caller's scratch, one row of block ids (with their kinds) per position.
//   3. prefill_refresh_kernel: every cache slot gets its block's K/V from the prompt
//      (the state after the prompt is the one the decode steps would have left).
//   4. prefill_attend_kernel: a CTA takes P consecutive positions of one unit, forms
//      the union of their selections and streams those blocks from the prompt's K and
//      V (TMA, 128-byte swizzle) through a ring of stages; every staged block is
//      attended by each of the P positions whose selection holds it (the tail block
//      of a position up to the position itself), with the decode attention's
//      tensor-core math per position.  Positions share every block they have in
//      common, so the K/V reads are shared P ways.
#include <cooperative_groups.h>

#include "attend_core.cuh"
#include "host.h"
#include "select_core.cuh"

namespace nosa {

using namespace selcore;

constexpr int kPfPositions = 4;        // positions per attention CTA
constexpr int kPfStages = 3;           // 32 KiB stages
constexpr int kPfMaxWords = 2048 / 32;  // block bitmap words per position (prompts of up to 131,072 tokens)
// a selection entry: block id in the low 12 bits, its kind (0 sink, 1 window, 2 query-aware,
// 3 query-agnostic) above; -1 pads
constexpr int kPfKindShift = 12;
constexpr int kPfBlockMask = (1 << kPfKindShift) - 1;

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------- 2. selections, in order
// Window logits of positions t0 .. t0 + np - 1 (np <= P), one CTA per unit: each 16-window tile
// of compressed keys is loaded once and multiplied with every position's q on the tensor cores
// (mma.sync m16n8k16, the group's heads as N = 8), so a tile's load serves P positions.  zp[p]
// [h][i] = z_{h,i} of position p, -inf for windows not complete at that position's T (nc[p]
// windows are).  Mst / Sst receive each position's per-head maximum and sum of exp.
template <int P>
__device__ __forceinline__ void score_positions(const LayerState& s, int u, const int (&nc)[P], int np,
                                                float* const (&zp)[P], const uint4 (&qf)[P][4],
                                                float (*Mst)[kMaxGroup], float (*Sst)[kMaxGroup],
                                                float (*cmax)[P][kMaxGroup]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gr = lane >> 2, t4 = lane & 3;
  const int G = s.G, wpc = s.score_wpc;
  const int nwarps = blockDim.x >> 5;
  const int tiles = wpc / (16 * nwarps);
  const int ncmax = nc[np - 1];  // the last position has the most windows
  const float scale = s.scale;
  float mx[P][2];
#pragma unroll
  for (int p = 0; p < P; ++p) mx[p][0] = mx[p][1] = -INFINITY;
  for (int t0 = 0; t0 < tiles; t0 += 2) {  // the loads of two tiles in flight together
    if ((warp * tiles + t0) * 16 >= ncmax) break;  // this warp's remaining tiles hold no complete window
    uint4 a[2][2][4];
#pragma unroll
    for (int tl = 0; tl < 2; ++tl)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int r = (warp * tiles + t0 + tl) * 16 + gr + 8 * hr;
        const bool ok = t0 + tl < tiles && r < ncmax;
        const uint16_t* kr = s.kt + ((size_t)u * s.nc_max + (ok ? r : 0)) * kHeadDim;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          a[tl][hr][c] = ok ? *reinterpret_cast<const uint4*>(kr + 32 * c + 8 * t4) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
    for (int tl = 0; tl < 2; ++tl) {
      if (t0 + tl >= tiles) break;
      const int wl0 = (warp * tiles + t0 + tl) * 16 + gr;
#pragma unroll
      for (int p = 0; p < P; ++p) {
        if (p >= np) break;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t* r0 = reinterpret_cast<const uint32_t*>(&a[tl][0][c]);
          const uint32_t* r1 = reinterpret_cast<const uint32_t*>(&a[tl][1][c]);
          const uint32_t* qq = reinterpret_cast<const uint32_t*>(&qf[p][c]);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const uint32_t af[4] = {r0[2 * hh], r1[2 * hh], r0[2 * hh + 1], r1[2 * hh + 1]};
            mma_16816(acc, af, qq[2 * hh], qq[2 * hh + 1]);
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int wl = wl0 + 8 * (j >> 1), h = 2 * t4 + (j & 1);
          const float z = wl < nc[p] ? acc[j] * scale : -INFINITY;
          zp[p][h * wpc + wl] = z;
          mx[p][j & 1] = fmaxf(mx[p][j & 1], z);
        }
      }
    }
  }
#pragma unroll
  for (int p = 0; p < P; ++p)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      mx[p][j] = fmaxf(mx[p][j], __shfl_xor_sync(0xffffffffu, mx[p][j], 4));
      mx[p][j] = fmaxf(mx[p][j], __shfl_xor_sync(0xffffffffu, mx[p][j], 8));
      mx[p][j] = fmaxf(mx[p][j], __shfl_xor_sync(0xffffffffu, mx[p][j], 16));
    }
  if (gr == 0)
#pragma unroll
    for (int p = 0; p < P; ++p) {
      cmax[warp][p][2 * t4] = mx[p][0];
      cmax[warp][p][2 * t4 + 1] = mx[p][1];
    }
  __syncthreads();
  if (tid < P * kMaxGroup) {
    const int p = tid / kMaxGroup, h = tid % kMaxGroup;
    float mm = -INFINITY;
    for (int w = 0; w < nwarps; ++w) mm = fmaxf(mm, cmax[w][p][h]);
    Mst[p][h] = mm;
  }
  __syncthreads();
  for (int ph = warp; ph < np * G; ph += nwarps) {  // sums of exp, one (position, head) per warp
    const int p = ph / G, h = ph % G;
    const float M = Mst[p][h];
    float e = 0.f;
    if (M > -INFINITY)
      for (int wl = lane; wl < nc[p]; wl += 32) e += expf(zp[p][h * wpc + wl] - M);
    e = warp_sum(e);
    if (lane == 0) Sst[p][h] = e;
  }
  __syncthreads();
}

// grid (1, U) in clusters of one CTA (the selector phases use the cluster API); 256 threads.
// q: [B][Hq][n][d]; hist: [U][n][cap] selection entries, -1 padded.  Positions are scored P at
// a time (score_positions), then selected one after the other: each position's selection needs
// the eviction state and slot map the previous one left.  Dynamic shared memory: the selector's
// region (whose logits array serves position 0) and P - 1 more logits arrays.
template <int P>
__global__ void __launch_bounds__(kScoreThreads, 1)
    prefill_select_kernel(LayerState s, const uint16_t* __restrict__ q, int16_t* __restrict__ hist, int n) {
  extern __shared__ __align__(16) unsigned char dsm[];
  __shared__ SelShared sh;
  __shared__ float cmax[kScoreWarps][P][kMaxGroup];
  __shared__ float Mst[P][kMaxGroup], Sst[P][kMaxGroup];
  cg::cluster_group cluster = cg::this_cluster();
  const int u = blockIdx.y, tid = threadIdx.x, lane = tid & 31;
  const Smem m = layout(dsm, s);
  const int G = s.G, wpc = s.score_wpc;
  float* zextra = reinterpret_cast<float*>(dsm + ((region_bytes(s) + 15) & ~size_t(15)));
  float* zp[P];
#pragma unroll
  for (int p = 0; p < P; ++p) zp[p] = p == 0 ? m.zs : zextra + (size_t)(p - 1) * kMaxGroup * wpc;
  pdl_wait();  // the bulk append before this kernel wrote the keys, scores and host store
  for (int t0 = 0; t0 < n; t0 += P) {
    const int np = min(P, n - t0);
    int nc[P];
    uint4 qf[P][4];
#pragma unroll
    for (int p = 0; p < P; ++p) {
      const int t = min(t0 + p, n - 1);
      nc[p] = geometry(t + 1, s.nw, s.sink).nc;
      // q of position t: head j of unit u is row (u * G + j) * n + t
      const int gr = lane >> 2, t4 = lane & 3;
      const uint16_t* qh = q + (((size_t)u * G + min(gr, G - 1)) * n + t) * kHeadDim;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        qf[p][c] = gr < G ? *reinterpret_cast<const uint4*>(qh + 32 * c + 8 * t4) : make_uint4(0, 0, 0, 0);
    }
    score_positions<P>(s, u, nc, np, zp, qf, Mst, Sst, cmax);
    for (int p = 0; p < np; ++p) {
      const int t = t0 + p, T = t + 1;
      const Geometry geo = geometry(T, s.nw, s.sink);
      const int my_slot_blk = leader_prefetch(s, u, geo.nb, geo.nb, m);
      if (tid < G) {
        sh.Mloc[tid] = Mst[p][tid];
        sh.Sloc[tid] = Sst[p][tid];
      }
      Smem mp = m;
      mp.zs = zp[p];
      pool_blocks(s, u, geo, 0, 1, mp, sh);  // opens with a barrier after the statistics above
      rank_local(s, geo, 0, 1, mp, sh);
      cluster.sync();
      cp_async_wait_all();
      // The context's pooled eviction scores cover the whole prompt.  At T a block pools only the
      // windows complete at T; for every block but the last two those are all its windows already.
      if (tid < 2) {
        const int b = geo.nb - 2 + tid;
        if (b >= 0) {
          const int lo = max(4 * b - 1, 0), hi = min(4 * b + 3, geo.nc - 1);
          float mx = -INFINITY;
          for (int i = lo; i <= hi; ++i) mx = fmaxf(mx, s.se_win[(size_t)u * s.nc_max + i]);
          m.sek[b] = mx;
        }
      }
      __syncthreads();
      int16_t* row = hist + ((size_t)u * n + t) * s.cap;
      const int nS = leader_select(s, u, geo, 1, mp, sh, my_slot_blk, true, [&](int pos, int b, int, bool, int, int kd) {
        row[pos] = (int16_t)(b | (kd << kPfKindShift));
      });
      for (int i = max(nS, 0) + tid; i < s.cap; i += blockDim.x) row[i] = -1;
      __syncthreads();  // this position's state (slots, eviction words) is read by the next one
    }
  }
}

// The same walk with one thread-block cluster of CS CTAs per unit, for layers with few units:
// CTA r scores windows [r * wpc, (r + 1) * wpc) of every position and pools and ranks the blocks
// it owns (the decode selector's phases, statistics and local winners through distributed
// shared memory between two cluster barriers); rank 0 then makes the selection on the state the
// previous position left while the other CTAs go on to score the next position.  Every
// cross-CTA read of a position happens between that position's two barriers, and no CTA writes
// the next position's statistics or winners before all have passed its first barrier.
__global__ void __launch_bounds__(kScoreThreads, 1)
    prefill_select_cluster_kernel(LayerState s, const uint16_t* __restrict__ q, int16_t* __restrict__ hist, int n) {
  extern __shared__ __align__(16) unsigned char dsm[];
  __shared__ SelShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank(), CS = (int)cluster.num_blocks();
  const int u = blockIdx.y, tid = threadIdx.x;
  const Smem m = layout(dsm, s);
  pdl_wait();  // the bulk append before this kernel wrote the keys, scores and host store
  for (int t = 0; t < n; ++t) {
    const int T = t + 1;
    const Geometry geo = geometry(T, s.nw, s.sink);
    int my_slot_blk = -1;
    if (rank == 0) my_slot_blk = leader_prefetch(s, u, geo.nb, geo.nb, m);
    uint4 qf[4];
    {  // q of position t: head j of unit u is row (u * G + j) * n + t
      const int lane = tid & 31, gr = lane >> 2, t4 = lane & 3;
      const uint16_t* qh = q + (((size_t)u * s.G + min(gr, s.G - 1)) * n + t) * kHeadDim;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        qf[c] = gr < s.G ? *reinterpret_cast<const uint4*>(qh + 32 * c + 8 * t4) : make_uint4(0, 0, 0, 0);
    }
    score_windows<2>(s, u, geo.nc, rank, m, sh, qf);
    cluster.sync();  // every CTA's statistics of this position are visible
    pool_blocks(s, u, geo, rank, CS, m, sh);
    rank_local(s, geo, rank, CS, m, sh);
    cluster.sync();  // the local winners have landed in rank 0; the statistics reads are done
    if (rank != 0) continue;
    cp_async_wait_all();
    // pooled eviction scores of the last two blocks as of T (windows complete at T only)
    if (tid < 2) {
      const int b = geo.nb - 2 + tid;
      if (b >= 0) {
        const int lo = max(4 * b - 1, 0), hi = min(4 * b + 3, geo.nc - 1);
        float mx = -INFINITY;
        for (int i = lo; i <= hi; ++i) mx = fmaxf(mx, s.se_win[(size_t)u * s.nc_max + i]);
        m.sek[b] = mx;
      }
    }
    __syncthreads();
    int16_t* row = hist + ((size_t)u * n + t) * s.cap;
    const int nS = leader_select(s, u, geo, CS, m, sh, my_slot_blk, true, [&](int pos, int b, int, bool, int, int kd) {
      row[pos] = (int16_t)(b | (kd << kPfKindShift));
    });
    for (int i = max(nS, 0) + tid; i < s.cap; i += blockDim.x) row[i] = -1;
    __syncthreads();  // this position's state (slots, eviction words) is read by the next one
  }
}

// ---------------------------------------------------------------- 3. cache refresh
// grid (cap, U), 256 threads: slot `slot` of unit u receives its block from the prompt's K/V
// (rows past the prompt zero), as the fetches of the decode steps would have left it.
__global__ void __launch_bounds__(256) prefill_refresh_kernel(LayerState s, const uint16_t* __restrict__ k,
                                                              const uint16_t* __restrict__ v, int n) {
  const int slot = blockIdx.x, u = blockIdx.y;
  pdl_wait();
  const int b = s.slot_blk[(size_t)u * s.cap + slot];
  if (b < 0 || b * kBlock >= n) return;
  uint16_t* dst = s.cache + ((size_t)u * s.cap + slot) * 2 * kBlockElems;
  for (int idx = threadIdx.x; idx < 2 * kBlock * 16; idx += blockDim.x) {
    const int kv = idx >> 10, r = (idx >> 4) & (kBlock - 1), c = idx & 15;
    const int tok = kBlock * b + r;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (tok < n) val = *reinterpret_cast<const uint4*>((kv ? v : k) + ((size_t)u * n + tok) * kHeadDim + 8 * c);
    *reinterpret_cast<uint4*>(dst + (size_t)kv * kBlockElems + r * kHeadDim + 8 * c) = val;
  }
}

// ---------------------------------------------------------------- 4. attention of every position
// grid (U, ceil(n / P)), 128 threads (four warps, 16 tokens of every block each).
template <int P>
__global__ void __launch_bounds__(kTeamThreads, 1)
    prefill_attend_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                          LayerState s, const uint16_t* __restrict__ q, uint16_t* __restrict__ out,
                          const int16_t* __restrict__ hist, int n) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[kPfStages];
  __shared__ uint32_t bm[P][kPfMaxWords];
  __shared__ int ublk[P * kMaxCacheSlots];
  __shared__ uint8_t umask[P * kMaxCacheSlots];
  __shared__ int n_union;
  __shared__ float wm[4][kMaxGroup], wl[4][kMaxGroup];
  __shared__ __align__(16) float sebuf[kPfStages][kBlock];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int u = blockIdx.x, t0 = blockIdx.y * P;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gr = lane >> 2, t4 = lane & 3;
  const int G = s.G, cap = s.cap;
  const int np = min(P, n - t0);
  const int nb_last = (t0 + np + kBlock - 1) / kBlock;  // blocks of the last position's context
  const int nbw = (nb_last + 31) / 32;
  const bool dma = s.dma_bias != 0;
  if (tid == 0) {
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
    for (int i = 0; i < kPfStages; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  pdl_wait();  // the selections, the prompt's K/V and (with the bias) the eviction scores
  for (int i = tid; i < P * kPfMaxWords; i += blockDim.x) bm[i / kPfMaxWords][i % kPfMaxWords] = 0u;
  __syncthreads();
  for (int idx = tid; idx < np * cap; idx += blockDim.x) {
    const int p = idx / cap, e = idx % cap;
    const int h = hist[((size_t)u * n + t0 + p) * cap + e];
    const int b = h & kPfBlockMask;
    if (h >= 0 && b < nb_last) atomicOr(&bm[p][b >> 5], 1u << (b & 31));
  }
  __syncthreads();
  if (warp == 0) {  // the union of the positions' selections, ascending, with a position mask each
    int base = 0;
    for (int w0 = 0; w0 < nbw; w0 += 32) {
      const int w = w0 + lane;
      uint32_t bits[P], uni = 0u;
#pragma unroll
      for (int p = 0; p < P; ++p) {
        bits[p] = w < nbw ? bm[p][w] : 0u;
        uni |= bits[p];
      }
      const int c = __popc(uni);
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int pos = base + incl - c;
      while (uni) {
        const int j = __ffs(uni) - 1;
        uni &= uni - 1u;
        uint8_t mk = 0;
#pragma unroll
        for (int p = 0; p < P; ++p) mk |= (uint8_t)(((bits[p] >> j) & 1u) << p);
        ublk[pos] = 32 * w + j;
        umask[pos] = mk;
        ++pos;
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) n_union = base;
  }
  // q fragments of every position (head gr of the group, 16 dims per k-step)
  uint32_t qb[P][8][2];
#pragma unroll
  for (int p = 0; p < P; ++p) {
    const int t = min(t0 + p, n - 1);
    const uint16_t* qh = q + (((size_t)u * G + min(gr, G - 1)) * n + t) * kHeadDim;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qb[p][ks][0] = gr < G ? *reinterpret_cast<const uint32_t*>(qh + 16 * ks + 2 * t4) : 0u;
      qb[p][ks][1] = gr < G ? *reinterpret_cast<const uint32_t*>(qh + 16 * ks + 2 * t4 + 8) : 0u;
    }
  }
  __syncthreads();
  const int nu = n_union;
  const uint32_t sbase = smem_u32(smem);
  auto issue = [&](int i) {  // union entry i into stage i % kPfStages
    if (i >= nu || tid != 0) return;
    const int st = i % kPfStages, b = ublk[i];
    const uint32_t dst = sbase + st * kStageBytes;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&bars[st], kStageBytes + (dma ? kBlock * 4 : 0));
    // stage layout [d half][K, V][64 tokens][64 dims]: four 8 KiB boxes
    tma_load_3d(dst, &tk, 0, kBlock * b, u, &bars[st]);
    tma_load_3d(dst + 8192, &tv, 0, kBlock * b, u, &bars[st]);
    tma_load_3d(dst + 16384, &tk, 64, kBlock * b, u, &bars[st]);
    tma_load_3d(dst + 24576, &tv, 64, kBlock * b, u, &bars[st]);
    if (dma) bulk_copy_g2s(smem_u32(sebuf[st]), s.se_tok + (size_t)u * s.se_stride + (size_t)kBlock * b, kBlock * 4,
                           &bars[st]);
  };
  for (int i = 0; i < kPfStages; ++i) issue(i);

  WarpAcc A[P];
#pragma unroll
  for (int p = 0; p < P; ++p) A[p].init();
  const float sl2 = s.scale * 1.4426950408889634f;
  const int tok0 = warp * 16;
  const int tk_k = tok0 + (lane & 7) + (((lane >> 3) & 1) << 3);
  const int ch_k = lane >> 4;
  const int tk_v = tok0 + (lane & 7) + ((lane >> 4) << 3);
  const int ch_v = (lane >> 3) & 1;
  bool bad = false;
  for (int i = 0; i < nu; ++i) {
    const int st = i % kPfStages, b = ublk[i];
    const uint8_t mk = umask[i];
    const bool okw = s.wait_limit >= 0 && mbar_wait_bounded(&bars[st], (uint32_t)((i / kPfStages) & 1), s.wait_limit);
    if (__syncthreads_or(!okw)) {
      if (tid == 0) atomicOr(s.err, kErrTimeout);
      bad = true;
      if (tid == 0)  // drain the copies still in flight before the shared memory goes away
        for (int j = i; j < min(i + kPfStages, nu); ++j)
          mbar_wait_bounded(&bars[j % kPfStages], (uint32_t)((j / kPfStages) & 1), kWaitCycles);
      break;
    }
    const uint32_t stg = sbase + st * kStageBytes;
#pragma unroll
    for (int p = 0; p < P; ++p) {
      if (!((mk >> p) & 1)) continue;
      const int Tp = t0 + p + 1;  // tokens in position p's context
      const int valid = min(Tp - kBlock * b, kBlock);
      if (tok0 >= valid) continue;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int dch = 2 * ks + ch_k;
        uint32_t a[4];
        ldsm_x4(a, swz(stg, dch >> 3, 0, tk_k, dch & 7));
        mma_16816(acc, a, qb[p][ks][0], qb[p][ks][1]);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[j] *= sl2;
      if (dma) {
        const float b0 = sebuf[st][tok0 + gr] * 1.4426950408889634f;
        const float b1 = sebuf[st][tok0 + gr + 8] * 1.4426950408889634f;
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
      WarpAcc& a_ = A[p];
      const float mn0 = fmaxf(a_.m0, mx0), mn1 = fmaxf(a_.m1, mx1);  // finite: token tok0 is valid
      const float al0 = exp2f(a_.m0 - mn0), al1 = exp2f(a_.m1 - mn1);
      const float p0 = exp2f(acc[0] - mn0), p1 = exp2f(acc[1] - mn1);
      const float p2 = exp2f(acc[2] - mn0), p3 = exp2f(acc[3] - mn1);
      a_.l0 = a_.l0 * al0 + p0 + p2;
      a_.l1 = a_.l1 * al1 + p1 + p3;
      a_.m0 = mn0;
      a_.m1 = mn1;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        a_.o[mt][0] *= al0;
        a_.o[mt][1] *= al1;
        a_.o[mt][2] *= al0;
        a_.o[mt][3] *= al1;
      }
      const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p0, p1));
      const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p2, p3));
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int dch = 2 * mt + ch_v;
        uint32_t a[4];
        ldsm_x4_trans(a, swz(stg, dch >> 3, 1, tk_v, dch & 7));
        mma_16816(a_.o[mt], a, pb0, pb1);
      }
    }
    __syncthreads();  // every warp is done with this stage
    issue(i + kPfStages);
  }
  __syncthreads();
  float* wo = reinterpret_cast<float*>(smem);  // [4 warps][8 heads][128], over the stages
#pragma unroll
  for (int p = 0; p < P; ++p) {
    if (bad) A[p].l0 = A[p].l1 = __int_as_float(0x7fc00000);  // a wait gave up: NaN outputs
    const int t = t0 + p;
    cta_partial<4>(A[p], wm, wl, wo, G, [&](int h, int x, float M, float L, float O) {
      if (t < n)
        out[(((size_t)u * G + h) * n + t) * kHeadDim + x] =
            __bfloat16_as_ushort(__float2bfloat16_rn(L > 0.f ? O / L : 0.f));
    });
    __syncthreads();  // wo, wm and wl are reused by the next position
  }
}

// ---------------------------------------------------------------- host side
size_t prefill_select_smem(const LayerState& s, int P) {
  return ((region_bytes(s) + 15) & ~size_t(15)) + (size_t)(P - 1) * kMaxGroup * s.score_wpc * sizeof(float);
}

static size_t prefill_attend_smem() { return 1024 + (size_t)kPfStages * kStageBytes; }

cudaError_t init_prefill_cluster(const LayerState& s) {
  cudaError_t e = cudaFuncSetAttribute(prefill_select_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)region_bytes(s));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(prefill_select_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

int prefill_cluster_active(const LayerState& s, int cs) {
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kScoreThreads);
  cfg.gridDim = dim3(cs, 1);
  cfg.dynamicSmemBytes = region_bytes(s);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int nc = 0;
  if (cudaOccupancyMaxActiveClusters(&nc, prefill_select_cluster_kernel, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return nc;
}

cudaError_t init_prefill(const LayerState& s, int P) {
  cudaError_t e = cudaFuncSetAttribute(prefill_attend_kernel<kPfPositions>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)prefill_attend_smem());
  const int sm = (int)prefill_select_smem(s, P);
  if (e == cudaSuccess)
    e = P == 4   ? cudaFuncSetAttribute(prefill_select_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm)
        : P == 2 ? cudaFuncSetAttribute(prefill_select_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm)
                 : cudaFuncSetAttribute(prefill_select_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
  return e;
}

int prefill_max_tokens() { return kPfMaxWords * 32 * kBlock; }

cudaError_t launch_prefill(const LayerState& s, int P, const CUtensorMap* tk, const CUtensorMap* tv,
                           const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* out, int16_t* hist,
                           int n, cudaStream_t st) {
  const dim3 block(kScoreThreads);
  cudaError_t e;
  if (s.score_chunks > 1) {  // a cluster per unit
    e = launch_ex(prefill_select_cluster_kernel, dim3(s.score_chunks, s.U), block, region_bytes(s), st, true,
                  s.score_chunks, s, q, hist, n);
  } else {
    const dim3 grid(1, s.U);
    const size_t sm = prefill_select_smem(s, P);
    e = P == 4   ? launch_ex(prefill_select_kernel<4>, grid, block, sm, st, true, 1, s, q, hist, n)
        : P == 2 ? launch_ex(prefill_select_kernel<2>, grid, block, sm, st, true, 1, s, q, hist, n)
                 : launch_ex(prefill_select_kernel<1>, grid, block, sm, st, true, 1, s, q, hist, n);
  }
  if (e != cudaSuccess) return e;
  e = launch_ex(prefill_refresh_kernel, dim3(s.cap, s.U), dim3(256), 0, st, true, 0, s, k, v, n);
  if (e != cudaSuccess) return e;
  return launch_ex(prefill_attend_kernel<kPfPositions>, dim3(s.U, (n + kPfPositions - 1) / kPfPositions),
                   dim3(kTeamThreads), prefill_attend_smem(), st, true, 0, *tk, *tv, s, q, out,
                   static_cast<const int16_t*>(hist), n);
}

}  // namespace nosa
