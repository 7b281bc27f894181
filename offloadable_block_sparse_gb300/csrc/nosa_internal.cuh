// Definitions shared by the kernels and the host code of libnosa.so: constants, the
// per-layer geometry, the layer state the kernels receive, and the launch helper.  The
// context object and the launchers are declared in host.h.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>
#include <vector>

#include "../../include/nosa.h"

namespace nosa {

constexpr int kHeadDim = 128;
constexpr int kBlock = 64;
constexpr int kCmpKernel = 32;
constexpr int kCmpStride = 16;
constexpr int kMaxGroup = 8;               // q heads per kv head handled by one MMA column tile
constexpr int kBlockElems = kBlock * kHeadDim;      // one K (or V) block: 8192 bf16 = 16 KiB
constexpr int kBlockBytes = 2 * kBlockElems * 2;    // K + V of one block: 32 KiB

// device error word bits
constexpr int kErrBounds = 1;
constexpr int kErrTimeout = 2;
constexpr int kErrCapacity = 4;

// one launch of the score/select kernel covers kScoreWarps * kScoreTiles * 16 windows per CTA
constexpr int kScoreThreads = 256;
constexpr int kScoreWarps = kScoreThreads / 32;
constexpr int kScoreTiles = 2;
constexpr int kWindowsPerCta = kScoreWarps * kScoreTiles * 16;

constexpr int kAttendThreads = 128;        // 4 warps, 16 tokens of every 64-token block each
constexpr int kAttendStages = 3;           // 32 KiB TMA stages per CTA
constexpr int kMaxBlocksPerCta = 64;       // split-K chunk: selected blocks per attend CTA
constexpr int kMaxCacheSlots = 256;        // cache slots per unit (sink + window + k_q + k_e)
constexpr int kPartStride = 2 + kHeadDim;  // (m, l, o[128]) per head in a split-K partial

constexpr int kGatherThreads = 512;
constexpr long long kWaitCycles = 2000000000LL;  // bounded device waits: about a second of SM clocks

// Per-layer derived quantities from the context length T (same formulas on host and device).
struct Geometry {
  int T, nb, nc, valid_tail, ws, ns;
};

__host__ __device__ inline Geometry geometry(int T, int nw, int sink) {
  Geometry g;
  g.T = T;
  g.nb = (T + kBlock - 1) / kBlock;
  g.nc = T < kCmpKernel ? 0 : (T - kCmpKernel) / kCmpStride + 1;
  g.valid_tail = T - kBlock * (g.nb - 1);
  g.ns = sink < g.nb ? sink : g.nb;
  int ws = g.nb - nw;
  g.ws = ws > g.ns ? ws : g.ns;
  return g;
}

// Device counters behind nosa_get_stats.
struct DevStats {
  unsigned long long selections;
  unsigned long long gamma_samples;
  unsigned long long gamma_num;   // sum of |D & S_prev|
  unsigned long long gamma_den;   // sum of |D|
  unsigned long long blocks_fetched;
  unsigned long long short_selections;
  unsigned int gamma_min_bits;    // float bits of the minimum gamma (non-negative floats order as ints)
  unsigned int pad;
};

// Pointers of one layer's state, offset by the host before each launch.
struct LayerState {
  int layer;
  int U;            // units of this layer
  int G;            // q heads per kv head
  int Hkv;
  int cap;          // blocks of one selection at most (sink + window + k_q + k_e): selection arrays
  int cslots;       // block cache slots per unit (cap or more)
  int nb_max, nc_max, T_max, ev_words, nw, sink, k_q, k_e, h;
  int se_stride;          // row stride of se_tok: nb_max * 64, so each block's scores start 256-byte aligned
  int dma_bias;           // attention logits get each token's eviction score added
  int unit_base;    // layer * U: first unit of this layer in context-wide arrays
  float scale;
  int* T;                 // device context length of this layer
  uint16_t* host_kv;      // device alias of the pinned store [U][nb_max][2][64][d]
  uint16_t* cache;        // [U][cslots][2][64][d]
  uint16_t* kt;           // [U][nc_max][d]
  uint16_t* kring;        // [U][32][d]
  float* se_tok;          // [U][se_stride]
  float* se_win;          // [U][nc_max]
  float* se_blk;          // [U][nb_max]
  int32_t* slot_blk;      // [U][cslots] block in each cache slot, -1 empty
  int32_t* last_used;     // [U][cslots] context length of the last selection holding the slot's block, -1 never
  int32_t* blk2slot;      // [U][nb_max]
  uint32_t* evicted;      // [U][ev_words]
  int32_t* sel;           // [U][cap]
  int32_t* sel_kind;      // [U][cap]
  int32_t* sel_slot;      // [U][cap]
  int32_t* sel_new;       // [U][cap] 1: the block had no slot before this selection (fetched)
  int32_t* n_sel;         // [U]
  int32_t* fetch;         // [U][cap][2]
  int32_t* n_fetch;       // [U]
  int32_t* gamma;         // [U][2]
  const float* W1;        // [Hkv][d][h]
  const float* W2;        // [Hkv][h]
  float* sq_blk;          // [U][nb_max] pooled query-aware scores of this layer's last selection
  // scratch shared by all layers (stream ordered)
  float* apart;           // [U][attend_chunks][kMaxGroup][kPartStride]
  unsigned int* tickets;  // [3][U]: append, score, attend
  DevStats* stats;
  int* err;
  int score_chunks;        // CTAs (one cluster) per unit in the selector
  int score_wpc;           // compressed windows per selector CTA (multiple of 128)
  int attend_chunks;       // split-K CTAs per unit in attend
  int attend_blocks_per_cta;
  int attend_mode;         // split-K merge: 0 ticket (global), 1 cluster (DSMEM), 2 merge kernel
  long long wait_limit;    // SM cycles a staged-block wait may take before it reports a timeout (<0: none)
  int test_bad_slot;       // test hook: publish one out-of-range slot (unit 0, first entry)
  int test_radix;          // test hook: the query-agnostic top-k always by warp radix select
};

}  // namespace nosa

namespace nosa {
// Launch through cudaLaunchKernelEx: optional programmatic dependent launch
// (the kernel overlaps its independent prologue with the previous kernel's
// tail; it calls griddepcontrol.wait before touching that kernel's results)
// and an optional cluster of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                      int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace nosa
