// Internal definitions shared by the translation units of libnosa.so.
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
  int cap, nb_max, nc_max, T_max, ev_words, nw, sink, k_q, k_e, h;
  int se_stride;          // row stride of se_tok: nb_max * 64, so each block's scores start 256-byte aligned
  int dma_bias;           // attention logits get each token's eviction score added
  int unit_base;    // layer * U: first unit of this layer in context-wide arrays
  float scale;
  int* T;                 // device context length of this layer
  uint16_t* host_kv;      // device alias of the pinned store [U][nb_max][2][64][d]
  uint16_t* cache;        // [U][cap][2][64][d]
  uint16_t* kt;           // [U][nc_max][d]
  uint16_t* kring;        // [U][32][d]
  float* se_tok;          // [U][se_stride]
  float* se_win;          // [U][nc_max]
  float* se_blk;          // [U][nb_max]
  int32_t* slot_blk;      // [U][cap]
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
  // scratch shared by all layers (stream ordered)
  float* sq_blk;          // [U][nb_max] pooled query-aware scores of the last selection
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
};

}  // namespace nosa

struct nosa_ctx {
  nosa_config cfg;
  nosa_sizes sz;
  int L, B, Hq, Hkv, G, d, U, h, nw, cap;
  cudaStream_t stream;
  int device;
  int num_sms;
  // pinned host store and its device alias
  uint16_t* host_kv;
  uint16_t* host_kv_dev;
  size_t host_layer_elems;
  // device state (all layers)
  void* dev_block;  // one allocation holding everything below
  uint16_t *cache, *kt, *kring;
  float *se_tok, *se_win, *se_blk, *W1, *W2;
  int32_t *slot_blk, *blk2slot, *sel, *sel_kind, *sel_slot, *sel_new, *n_sel, *fetch, *n_fetch, *gamma;
  uint32_t* evicted;
  int *T, *err;
  nosa::DevStats* stats;
  // scratch
  float *sq_blk, *apart;
  unsigned int* tickets;
  int score_chunks, score_wpc, attend_chunks, attend_blocks_per_cta, attend_mode, gather_ctas;
  // fused decode kernel (nosa_step): cluster size (0: off, three kernels instead), windows per
  // scoring CTA, attention stages per team
  int dec_cs, dec_wpc, dec_nst, dec_teams;
  // staging buffers for host-pointer calls
  uint16_t *stage_q, *stage_k, *stage_v, *stage_out;
  uint16_t *step_q, *step_k, *step_v, *step_out;  // every layer's inputs and outputs (nosa_step_host_all)
  size_t stage_tok_cap;   // tokens per unit the bulk staging buffers hold
  uint16_t *bulk_k, *bulk_v;
  // TMA descriptor of the block cache (4-D: d, token, K/V, flat slot)
  CUtensorMap tmap_cache;
  // host mirrors
  std::vector<int> T_host;
  std::vector<int> sel_T;   // T at the last selection (-1: none), host view
  std::vector<int> fetch_T; // T at the last nosa_fetch (-1: none): attend fetches itself otherwise
  int failed;               // latched nosa_status of a device-side error
  // forecast pipeline: prefetch stream, fork event, one "prefetched" event per layer and whether
  // the layer's stream still has to wait for it
  cudaStream_t pref_stream;
  cudaEvent_t ev_fork;
  std::vector<cudaEvent_t> ev_pref;
  std::vector<char> pref_pending;
};

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

LayerState layer_state(nosa_ctx* c, int layer);
// pdl: launch as a programmatic dependent of the previous kernel in the stream
cudaError_t launch_append_one(const LayerState& s, const uint16_t* k, const uint16_t* v, bool pdl, cudaStream_t st);
cudaError_t launch_append_bulk(const LayerState& s, const uint16_t* k, const uint16_t* v, int T_old,
                               int n, cudaStream_t st);
// ahead = 1: forecast selection / its gather, made before the next token is appended
// knew/vnew (ahead 0 only): the kernel also appends the step's token (the step path).
cudaError_t launch_score_select(const LayerState& s, const uint16_t* q, bool pdl, cudaStream_t st, int ahead = 0,
                                const uint16_t* knew = nullptr, const uint16_t* vnew = nullptr);
cudaError_t launch_gather(const LayerState& s, int ctas, cudaStream_t st, int ahead = 0);
// fused_fetch != 0: blocks marked in sel_new are copied from the pinned host
// store by the attend CTAs themselves (and written back to their slots), so no
// separate gather launch is needed.
cudaError_t launch_attend(const LayerState& s, const CUtensorMap* tmap, const uint16_t* q, uint16_t* out,
                          int fused_fetch, bool pdl, cudaStream_t st);
// merges s.attend_chunks split-K partials per unit from s.apart into out (at most 256 chunks)
cudaError_t launch_attend_merge(const LayerState& s, uint16_t* out, cudaStream_t st);
size_t score_select_smem(const LayerState& s);
// one-time kernel attributes (dynamic shared memory limits), called by nosa_create
cudaError_t init_append(const LayerState& s);
cudaError_t init_score_select(const LayerState& s);
cudaError_t init_attend();
int attend_max_cluster();
// fused decode step of one layer (append + select + fetch + attend); s carries the fused
// kernel's cluster size and windows per CTA in score_chunks / score_wpc
LayerState decode_state(nosa_ctx* c, int layer);
// teams: attention workers (four warps each) per CTA, 1 or 2; nst: stages per worker
size_t decode_smem_bytes(const LayerState& s, int teams, int nst);
cudaError_t init_decode(const LayerState& s, int teams, int nst);
int decode_active_clusters(const LayerState& s, int teams, int nst, int cs);
cudaError_t launch_decode(const LayerState& s, const CUtensorMap* tmap, const uint16_t* q, const uint16_t* k,
                          const uint16_t* v, uint16_t* out, int teams, int nst, bool pdl, cudaStream_t st);
}  // namespace nosa
