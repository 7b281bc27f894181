// a2-a4 selector kernel: the scorer and two-part selector phases (shared with
// the fused decode kernel) composed with cluster barriers between them.
#include "select_core.cuh"

namespace nosa {

using namespace selcore;

// grid (cluster size, U) with clusters (cluster size, 1, 1); 256 threads; dynamic
// shared memory selcore::region_bytes.  ahead = 1: a forecast selection made before
// the next token is appended (SparDA summary: one layer ahead) -- blocks, sink,
// window and candidates of T + 1, scores over the windows complete at T; q is then
// one forecast vector per unit (s.G = 1).
__global__ void __launch_bounds__(kScoreThreads) score_select_kernel(LayerState s, const uint16_t* __restrict__ q,
                                                                     int ahead) {
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
  const int T = *s.T;
  Geometry geo = geometry(T + ahead, s.nw, s.sink);
  geo.nc = geometry(T, s.nw, s.sink).nc;  // windows that exist now
  int my_slot_blk = -1;
  if (rank == 0) my_slot_blk = leader_prefetch(s, u, geo.nb, geo.nb, m);
  score_windows<2>(s, u, geo.nc, rank, m, sh, qf);
  cluster.sync();  // every CTA's statistics are visible
  pool_blocks(s, u, geo, rank, CS, m, sh);
  rank_local(s, geo, rank, CS, m, sh);
  cluster.sync();  // the local winners have landed in the leader; remote reads are done
  if (rank != 0) return;
  cp_async_wait_all();  // the leader's early copies (pooled s^e, slot map, eviction words)
  leader_select(s, u, geo, CS, m, sh, my_slot_blk, true, NoDeal{});
}

size_t score_select_smem(const LayerState& s) { return region_bytes(s); }

cudaError_t init_score_select(const LayerState& s) {
  return cudaFuncSetAttribute(score_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)score_select_smem(s));
}

cudaError_t launch_score_select(const LayerState& s, const uint16_t* q, bool pdl, cudaStream_t st, int ahead) {
  return launch_ex(score_select_kernel, dim3(s.score_chunks, s.U), dim3(kScoreThreads), score_select_smem(s), st,
                   pdl, s.score_chunks, s, q, ahead);
}

}  // namespace nosa
