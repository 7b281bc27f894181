// Fused decode step of one layer: a1 append, a2 score, a3 select, a4 set
// difference, a5 fetch and a6 attend in one kernel, one thread-block cluster of
// CS CTAs per unit; a CTA is kTeams (1 or 2) teams of four warps, one attention
// worker each.
//
//   prologue  wait for the previous kernel (the inputs may be its outputs), read
//             the context length, q, and take a ticket; the last CTA of the grid
//             advances the length.
//   a1        the last CTA of the cluster (the one with the fewest windows to
//             score) appends the token; the CTA scoring the window this token
//             completes computes that window's compressed key itself, so no
//             CTA waits for the append before scoring.
//   a2-a4     the selector phases with cluster barriers between them (scores and
//             statistics through distributed shared memory, local top-k_q per
//             CTA, pushed to every CTA).  Every CTA then runs the selection on
//             the same inputs and reaches the same result; rank 0 alone stores
//             the unit's selection state, and each CTA keeps its own workers'
//             shares of the list, so no list crosses the cluster.
//   a5-a6     every team is one split-K worker (the attention core: TMA ring
//             over the block cache, blocks still on the host copied by cp.async
//             and written to their new cache slot); the unit's selected blocks
//             are dealt round-robin to the kTeams*CS workers, blocks without a
//             slot first; the warps' partials are merged in shared memory and
//             the CTAs' partials through distributed shared memory.
// The selector's shared memory and the attention stages alias: a CTA's own selection
// is complete (CTA barrier) before its stages are loaded, and no CTA reads another's
// selector memory after the second cluster barrier.
#include <algorithm>

#include "append_core.cuh"
#include "attend_core.cuh"
#include "host.h"
#include "select_core.cuh"

namespace nosa {

using namespace selcore;

constexpr int kDecodeMaxStages = 6;   // per team

template <int kTeams>
__global__ void __launch_bounds__(kTeamThreads * kTeams, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmap, LayerState s, const uint16_t* __restrict__ q,
                  const uint16_t* __restrict__ knew, const uint16_t* __restrict__ vnew, uint16_t* __restrict__ out,
                  int nst) {
  constexpr int kThreads = kTeamThreads * kTeams;
  constexpr int kSlots = kThreads;  // the leader's slot scan: one thread per cache slot
  extern __shared__ unsigned char smem_raw[];
  __shared__ SelShared sh;
  __shared__ __align__(8) uint64_t bars[kTeams][kDecodeMaxStages];
  __shared__ int w_blk[kTeams][kSlots], w_slot[kTeams][kSlots], w_new[kTeams][kSlots];
  __shared__ float wm[4 * kTeams][kMaxGroup], wl[4 * kTeams][kMaxGroup];
  __shared__ float cp_m[kMaxGroup], cp_l[kMaxGroup], cp_o[kMaxGroup][kHeadDim];
  __shared__ __align__(16) float sebuf[kTeams][kDecodeMaxStages][kBlock];  // staged blocks' eviction scores
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank(), CS = (int)cluster.num_blocks();
  const int u = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int team = warp >> 2, ttid = tid & (kTeamThreads - 1);
  const int G = s.G;
  const Smem m = layout(smem, s);

  if (tid == 0) {
    prefetch_tmap(&tmap);
    for (int t = 0; t < kTeams; ++t)
      for (int i = 0; i < nst; ++i) mbar_init(&bars[t][i], 1);
    fence_mbar_init();
  }
  // q, k_new and v_new may be written by the previous kernel: wait before reading anything
  pdl_wait();
  pdl_launch_dependents();  // the next kernel may launch; it waits for this one before its reads
  const int p = *s.T;       // position of the new token
  if (p >= s.T_max) {       // every CTA sees the same p and returns; the length stays
    if (tid == 0 && rank == 0 && u == 0) atomicOr(s.err, kErrCapacity);
    return;
  }
  const int T = p + 1;
  const Geometry geo = geometry(T, s.nw, s.sink);
  if (tid == 0) {  // this CTA has read the length: the last one to get here advances it
    unsigned int* tk = s.tickets + 3 * s.U;
    if (atomicAdd(tk, 1u) == gridDim.x * gridDim.y - 1) {
      *tk = 0;
      *s.T = T;
    }
  }
  uint4 qf[4];
  load_q(qf, q, u, G);
  uint32_t qb[8][2];
  load_q_frags(qb, q, u, G, lane);

  // ---------------- a1: append; the window completed by this token gets its key from its scorer
  const bool window_done = T >= kCmpKernel && (T - kCmpKernel) % kCmpStride == 0;
  const int wi = window_done ? (T - kCmpKernel) / kCmpStride : -1;
  // pooled s^e of the last two blocks may change in this step (a completed window overlaps
  // only them); the leader reads those after the append, the rest now
  const int nb_se = max(min(geo.ws, geo.nb - 2), 0);
  const int my_slot_blk = leader_prefetch(s, u, geo.nb, nb_se, m);  // every CTA selects
  // the window's scorer, and the next CTA, which scores it as the window before its range,
  // both compute its key (the same bits) before they read it
  if (window_done && (wi / s.score_wpc == rank || wi == rank * s.score_wpc - 1)) window_key(s, u, p, wi, knew);
  if (rank == CS - 1) {
    append_token<kThreads>(s, u, p, knew, vnew, false);
    fence_proxy_async_global();  // the token's cache row is read by TMA later in this kernel
  }
  __syncthreads();  // the window key written above is read by this CTA's scorer

  // ---------------- a2-a4: selector phases
  score_windows<4>(s, u, geo.nc, rank, m, sh, qf);
  if (rank == CS - 1) __threadfence_system();  // the token's host-store row, copied by other CTAs below
  cluster.sync();  // every CTA's statistics are visible
  // pooled s^e of the last two blocks (written by the append before the barrier above): loaded
  // now, so that the load lands while the CTAs pool and rank
  const int b_se = nb_se + tid;
  const float se_patch = (tid < 2 && b_se < geo.ws) ? s.se_blk[(size_t)u * s.nb_max + b_se] : 0.f;
  pool_blocks(s, u, geo, rank, CS, m, sh);
  rank_local(s, geo, rank, CS, m, sh, true);
  cluster.sync();  // every CTA holds all local winners; the append's pooled s^e are visible

  // ---------------- a5-a6: every CTA selects (rank 0 also stores the unit's selection state)
  // and keeps its workers' shares: position dp of the dealing order (blocks without a slot
  // first) goes to worker dp % NW
  cp_async_wait_all();  // the early copies (pooled s^e, slot map, eviction words)
  if (tid < 2 && b_se < geo.ws) m.sek[b_se] = se_patch;  // read by the selection after its first barrier
  const int NW = kTeams * CS, wkr = kTeams * rank + team;  // workers of the unit, this one
  const int total_S = leader_select(s, u, geo, CS, m, sh, my_slot_blk, rank == 0,
                                    [&](int pos, int b, int slot, bool isnew, int dp, int) {
                                      const int w = dp % NW;
                                      if (w / kTeams != rank || dp >= s.cap) return;
                                      if (slot < 0 || slot >= s.cslots) {
                                        atomicOr(s.err, kErrBounds);
                                        slot = 0;  // keep the copy in bounds; the result is flagged
                                      }
                                      const int t = w % kTeams, i = dp / NW;
                                      w_blk[t][i] = b;
                                      w_slot[t][i] = slot;
                                      w_new[t][i] = isnew ? 1 : 0;
                                    });
  // a selection larger than the cache is an error (flagged by the selection): attend nothing
  const int nsel = total_S <= s.cap ? total_S : 0;
  const int my_n = wkr < nsel ? (nsel - wkr + NW - 1) / NW : 0;
  __syncthreads();  // the workers' lists are complete

  WarpAcc A;
  A.init();
  const uint32_t sbase = smem_u32(smem) + (uint32_t)(team * nst * kStageBytes);
  attend_worker(&tmap, s, geo, u, qb, w_blk[team], w_slot[team], w_new[team], my_n, sbase, bars[team], nst,
                &sebuf[team][0][0], Team{kTeams == 1 ? 0u : 1u + (uint32_t)team}, ttid, A);
  __syncthreads();  // every copy has landed (or was drained): the stages can hold the warp partials

  float* wo = reinterpret_cast<float*>(smem);  // [warps][8 heads][128]
  cta_partial<4 * kTeams>(A, wm, wl, wo, G, [&](int h, int x, float M, float L, float O) {
    if (x == 0) {
      cp_m[h] = M;
      cp_l[h] = L;
    }
    cp_o[h][x] = O;
  });
  // every CTA of the unit merges the heads h = rank, rank + CS, ... from all CTAs' partials,
  // one output element per thread
  cluster.sync();
  {
    const int nh = (G - rank + CS - 1) / CS;
    for (int idx = tid; idx < nh * kHeadDim; idx += blockDim.x) {
      const int h = rank + CS * (idx >> 7), x = idx & (kHeadDim - 1);
      float mr[8], M = -INFINITY;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        mr[r] = r < CS ? *cluster.map_shared_rank(&cp_m[h], r) : -INFINITY;
        M = fmaxf(M, mr[r]);
      }
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        if (r < CS && mr[r] > -INFINITY) {
          const float f = exp2f(mr[r] - M);
          L += *cluster.map_shared_rank(&cp_l[h], r) * f;
          O += *cluster.map_shared_rank(&cp_o[h][x], r) * f;
        }
      }
      const float res = L > 0.f ? O / L : 0.f;
      out[((size_t)u * G + h) * kHeadDim + x] = __bfloat16_as_ushort(__float2bfloat16_rn(res));
    }
  }
  cluster.sync();  // keep every CTA's shared memory alive until all remote reads are done
}

size_t decode_smem_bytes(const LayerState& s, int teams, int nst) {
  const size_t stages = (size_t)teams * nst * kStageBytes;
  return 1024 + std::max(region_bytes(s), stages);
}

template <int kTeams>
static cudaError_t set_decode_attrs(const LayerState& s, int nst) {
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<kTeams>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)decode_smem_bytes(s, kTeams, nst));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_kernel<kTeams>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

cudaError_t init_decode(const LayerState& s, int teams, int nst) {
  return teams == 2 ? set_decode_attrs<2>(s, nst) : set_decode_attrs<1>(s, nst);
}

// Clusters of `cs` decode CTAs that the device can hold at once (0: none).
int decode_active_clusters(const LayerState& s, int teams, int nst, int cs) {
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kTeamThreads * teams);
  cfg.gridDim = dim3(cs, 1);
  cfg.dynamicSmemBytes = decode_smem_bytes(s, teams, nst);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  const cudaError_t e = teams == 2 ? cudaOccupancyMaxActiveClusters(&n, decode_kernel<2>, &cfg)
                                   : cudaOccupancyMaxActiveClusters(&n, decode_kernel<1>, &cfg);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_decode(const LayerState& s, const CUtensorMap* tmap, const uint16_t* q, const uint16_t* k,
                          const uint16_t* v, uint16_t* out, int teams, int nst, bool pdl, cudaStream_t st) {
  const size_t smem = decode_smem_bytes(s, teams, nst);
  const dim3 grid(s.score_chunks, s.U), block(kTeamThreads * teams);
  if (teams == 2)
    return launch_ex(decode_kernel<2>, grid, block, smem, st, pdl, s.score_chunks, *tmap, s, q, k, v, out, nst);
  return launch_ex(decode_kernel<1>, grid, block, smem, st, pdl, s.score_chunks, *tmap, s, q, k, v, out, nst);
}

}  // namespace nosa
