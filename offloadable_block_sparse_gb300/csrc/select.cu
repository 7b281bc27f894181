// a2-a4 selector kernel: the scorer and two-part selector phases (shared with
// the fused decode kernel) composed with cluster barriers between them; in a step
// (nosa_step) it also runs a1, the append of the token, as the fused kernel does.
#include "append_core.cuh"
#include "host.h"
#include "select_core.cuh"

namespace nosa {

using namespace selcore;

// grid (cluster size, U) with clusters (cluster size, 1, 1); 256 threads; dynamic
// shared memory selcore::region_bytes.  ahead = 1: a forecast selection made before
// the next token is appended (SparDA summary: one layer ahead) -- blocks, sink,
// window and candidates of T + 1, scores over the windows complete at T; q is then
// one forecast vector per unit (s.G = 1).  With knew/vnew (ahead = 0) the kernel first
// appends the token: the last CTA of each cluster appends it, the CTA scoring the window
// it completes (and its right neighbour) computes that window's key, the last CTA of the
// grid to take a ticket advances T, and the leader reads the pooled s^e of the last two
// blocks (which the append may change) after the cluster barriers.
__global__ void __launch_bounds__(kScoreThreads) score_select_kernel(LayerState s, const uint16_t* __restrict__ q,
                                                                     int ahead, const uint16_t* __restrict__ knew,
                                                                     const uint16_t* __restrict__ vnew) {
  extern __shared__ __align__(16) unsigned char dsm[];
  __shared__ SelShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank(), CS = (int)cluster.num_blocks();
  const int u = blockIdx.y;
  const Smem m = layout(dsm, s);
  pdl_wait();               // q may come from a kernel before the append; keys and scores from the append
  pdl_launch_dependents();  // the attention kernel may start its own prologue
  uint4 qf[4];
  load_q(qf, q, u, s.G);
  const bool app = knew != nullptr;  // this step's append runs here
  int T = *s.T;
  if (app) {
    if (T >= s.T_max) {  // every CTA sees the same length and returns; nothing changes
      if (threadIdx.x == 0 && rank == 0 && u == 0) atomicOr(s.err, kErrCapacity);
      return;
    }
    T += 1;
    if (threadIdx.x == 0) {  // this CTA has read the length: the last one to get here advances it
      unsigned int* tk = s.tickets + 3 * s.U;
      if (atomicAdd(tk, 1u) == gridDim.x * gridDim.y - 1) {
        *tk = 0;
        *s.T = T;
      }
    }
  }
  Geometry geo = geometry(T + ahead, s.nw, s.sink);
  geo.nc = geometry(T, s.nw, s.sink).nc;  // windows that exist now
  // pooled s^e of the last two blocks may change with the append: the leader reads those later
  const int nb_se = app ? max(min(geo.ws, geo.nb - 2), 0) : geo.nb;
  int my_slot_blk = -1;
  if (rank == 0) my_slot_blk = leader_prefetch(s, u, geo.nb, nb_se, m);
  if (app) {
    const int p = T - 1;
    const bool window_done = T >= kCmpKernel && (T - kCmpKernel) % kCmpStride == 0;
    const int wi = window_done ? (T - kCmpKernel) / kCmpStride : -1;
    if (window_done && (wi / s.score_wpc == rank || wi == rank * s.score_wpc - 1)) window_key(s, u, p, wi, knew);
    if (rank == CS - 1) append_token<kScoreThreads>(s, u, p, knew, vnew, false);
    __syncthreads();  // the window key written above is read by this CTA's scorer
  }
  score_windows<2>(s, u, geo.nc, rank, m, sh, qf);
  cluster.sync();  // every CTA's statistics are visible
  pool_blocks(s, u, geo, rank, CS, m, sh);
  rank_local(s, geo, rank, CS, m, sh);
  cluster.sync();  // the local winners have landed in the leader; remote reads are done
  if (rank != 0) return;
  cp_async_wait_all();  // the leader's early copies (pooled s^e, slot map, eviction words)
  if (app) {
    if (threadIdx.x < 2) {
      const int b = nb_se + threadIdx.x;
      if (b < geo.ws) m.sek[b] = s.se_blk[(size_t)u * s.nb_max + b];  // after the append's update
    }
    __syncthreads();
  }
  leader_select(s, u, geo, CS, m, sh, my_slot_blk, true, NoDeal{});
}

size_t score_select_smem(const LayerState& s) { return region_bytes(s); }

cudaError_t init_score_select(const LayerState& s) {
  return cudaFuncSetAttribute(score_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)score_select_smem(s));
}

cudaError_t launch_score_select(const LayerState& s, const uint16_t* q, bool pdl, cudaStream_t st, int ahead,
                                const uint16_t* knew, const uint16_t* vnew) {
  return launch_ex(score_select_kernel, dim3(s.score_chunks, s.U), dim3(kScoreThreads), score_select_smem(s), st,
                   pdl, s.score_chunks, s, q, ahead, knew, vnew);
}

}  // namespace nosa
