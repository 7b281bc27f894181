// C ABI of libnosa.so: configuration, allocation, launches and error latching.
// The entry points and their contracts are documented in include/nosa.h.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <new>

#include "host.h"

using namespace nosa;

namespace {

#define CK(call)                              \
  do {                                        \
    if ((call) != cudaSuccess) {              \
      (void)cudaGetLastError();               \
      return NOSA_ERR_CUDA;                   \
    }                                         \
  } while (0)

inline int cdiv(long long a, long long b) { return (int)((a + b - 1) / b); }

__global__ void fill_f32(float* p, size_t n, float v) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) p[i] = v;
}

__global__ void copy_i32(int32_t* dst, const int32_t* src, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

struct Derived {
  int U, G, nw, cap, cs, nb_max, nc_max, ev_words, h;
};

Derived derive(const nosa_config* c) {
  Derived d;
  d.U = c->batch * c->num_kv_heads;
  d.G = c->num_q_heads / c->num_kv_heads;
  d.nw = c->window_tokens / c->block_size;
  d.cap = c->sink_blocks + d.nw + c->k_q + c->k_e;
  // the block cache: twice a selection by default, so that blocks leaving the selection stay
  // cached for a while (a block the query-aware part picks again is then not fetched again)
  d.cs = c->cache_slots > 0 ? c->cache_slots : std::min(2 * d.cap, kMaxCacheSlots);
  d.nb_max = cdiv(c->max_context, kBlock);
  d.nc_max = c->max_context < kCmpKernel ? 0 : (c->max_context - kCmpKernel) / kCmpStride + 1;
  d.ev_words = cdiv(d.nb_max, 32);
  d.h = c->evict_hidden;
  return d;
}

nosa_status check_ctx(nosa_ctx* c, int layer) {
  if (!c) return NOSA_ERR_INVALID_ARG;
  if (c->failed) return NOSA_ERR_STATE;
  if (layer < 0 || layer >= c->L) return NOSA_ERR_INVALID_ARG;
  return NOSA_OK;
}

nosa_status err_to_status(int e) {
  if (e & kErrBounds) return NOSA_ERR_BOUNDS;
  if (e & kErrTimeout) return NOSA_ERR_TIMEOUT;
  if (e & kErrCapacity) return NOSA_ERR_CAPACITY;
  return NOSA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

void free_ctx(nosa_ctx* c) {
  void* dev[] = {c->cache, c->kt, c->kring, c->se_tok, c->se_win, c->se_blk, c->W1, c->W2, c->slot_blk, c->last_used,
                 c->blk2slot, c->sel, c->sel_kind, c->sel_slot, c->sel_new, c->n_sel, c->fetch, c->n_fetch, c->gamma,
                 c->evicted, c->T, c->err, c->stats, c->sq_blk, c->apart, c->tickets,
                 c->stage_q, c->stage_k, c->stage_v, c->stage_out, c->bulk_k, c->bulk_v,
                 c->step_q, c->step_k, c->step_v, c->step_out};
  for (void* p : dev)
    if (p) cudaFree(p);
  if (c->host_kv) cudaFreeHost(c->host_kv);
  for (cudaEvent_t e : c->ev_sel)
    if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : c->ev_pref)
    if (e) cudaEventDestroy(e);
  if (c->ev_fork) cudaEventDestroy(c->ev_fork);
  if (c->pref_stream) cudaStreamDestroy(c->pref_stream);
  if (c->sel_stream) cudaStreamDestroy(c->sel_stream);
  delete c;
}

}  // namespace

namespace nosa {
LayerState layer_state(nosa_ctx* c, int l) {
  LayerState s;
  const Derived d = derive(&c->cfg);
  const size_t U = d.U;
  s.layer = l;
  s.U = d.U;
  s.G = d.G;
  s.Hkv = c->Hkv;
  s.cap = d.cap;
  s.cslots = d.cs;
  s.nb_max = d.nb_max;
  s.nc_max = std::max(d.nc_max, 1);
  s.T_max = c->cfg.max_context;
  s.ev_words = d.ev_words;
  s.nw = d.nw;
  s.sink = c->cfg.sink_blocks;
  s.k_q = c->cfg.k_q;
  s.k_e = c->cfg.k_e;
  s.h = d.h;
  s.unit_base = l * d.U;
  s.scale = c->cfg.softmax_scale > 0.f ? c->cfg.softmax_scale : 1.f / sqrtf((float)kHeadDim);
  const size_t lu = (size_t)l * U;
  s.T = c->T + l;
  s.host_kv = c->host_kv_dev + lu * d.nb_max * 2 * kBlockElems;
  s.cache = c->cache + lu * d.cs * 2 * kBlockElems;
  s.kt = c->kt + lu * s.nc_max * kHeadDim;
  s.kring = c->kring + lu * 32 * kHeadDim;
  s.se_stride = d.nb_max * kBlock;
  s.se_tok = c->se_tok + lu * s.se_stride;
  s.se_win = c->se_win + lu * s.nc_max;
  s.se_blk = c->se_blk + lu * d.nb_max;
  s.slot_blk = c->slot_blk + lu * d.cs;
  s.last_used = c->last_used + lu * d.cs;
  s.blk2slot = c->blk2slot + lu * d.nb_max;
  s.evicted = c->evicted + lu * d.ev_words;
  s.sel = c->sel + lu * d.cap;
  s.sel_kind = c->sel_kind + lu * d.cap;
  s.sel_slot = c->sel_slot + lu * d.cap;
  s.sel_new = c->sel_new + lu * d.cap;
  s.n_sel = c->n_sel + lu;
  s.fetch = c->fetch + lu * d.cap * 2;
  s.n_fetch = c->n_fetch + lu;
  s.gamma = c->gamma + lu * 2;
  s.W1 = c->W1 + (size_t)l * c->Hkv * kHeadDim * d.h;
  s.W2 = c->W2 + (size_t)l * c->Hkv * d.h;
  s.sq_blk = c->sq_blk + lu * d.nb_max;
  s.apart = c->apart;
  s.tickets = c->tickets;
  s.stats = c->stats;
  s.err = c->err;
  s.score_chunks = c->score_chunks;
  s.score_wpc = c->score_wpc;
  s.attend_chunks = c->attend_chunks;
  s.attend_blocks_per_cta = c->attend_blocks_per_cta;
  s.attend_mode = c->attend_mode;
  s.wait_limit = (c->cfg.flags & NOSA_F_TEST_ZERO_WAIT) ? -1 : kWaitCycles;
  s.test_bad_slot = (c->cfg.flags & NOSA_F_TEST_BAD_SLOT) ? 1 : 0;
  s.test_radix = (c->cfg.flags & NOSA_F_TEST_RADIX_TOPK) ? 1 : 0;
  s.dma_bias = (c->cfg.flags & NOSA_F_DMA_BIAS) ? 1 : 0;
  return s;
}

LayerState decode_state(nosa_ctx* c, int layer) {
  LayerState s = layer_state(c, layer);
  s.score_chunks = c->dec_cs;
  s.score_wpc = c->dec_wpc;
  return s;
}
}  // namespace nosa

extern "C" {

const char* nosa_status_string(nosa_status s) {
  switch (s) {
    case NOSA_OK: return "ok";
    case NOSA_ERR_INVALID_ARG: return "invalid argument";
    case NOSA_ERR_OOM: return "device out of memory";
    case NOSA_ERR_HOST_ALLOC: return "pinned host allocation failed";
    case NOSA_ERR_CUDA: return "CUDA runtime error";
    case NOSA_ERR_CAPACITY: return "context capacity exceeded";
    case NOSA_ERR_TIMEOUT: return "device-side wait timed out";
    case NOSA_ERR_BOUNDS: return "device-side bounds check failed";
    case NOSA_ERR_STATE: return "call out of order or context failed";
  }
  return "unknown status";
}

nosa_status nosa_validate_config(const nosa_config* c) {
  if (!c || c->struct_size != sizeof(nosa_config)) return NOSA_ERR_INVALID_ARG;
  if (c->num_layers < 1 || c->batch < 1 || c->num_kv_heads < 1 || c->num_q_heads < 1) return NOSA_ERR_INVALID_ARG;
  if (c->num_q_heads % c->num_kv_heads) return NOSA_ERR_INVALID_ARG;
  const int G = c->num_q_heads / c->num_kv_heads;
  if (G < 1 || G > kMaxGroup) return NOSA_ERR_INVALID_ARG;
  if (c->head_dim != kHeadDim || c->block_size != kBlock) return NOSA_ERR_INVALID_ARG;
  if (c->cmp_kernel != kCmpKernel || c->cmp_stride != kCmpStride) return NOSA_ERR_INVALID_ARG;
  if (c->k_q < 0 || c->k_e < 0 || c->sink_blocks < 0) return NOSA_ERR_INVALID_ARG;
  if (c->window_tokens < 0 || c->window_tokens % kBlock) return NOSA_ERR_INVALID_ARG;
  if (c->max_context < 1 || c->max_context > 262144) return NOSA_ERR_INVALID_ARG;
  if (c->evict_hidden < 32 || c->evict_hidden > 256 || c->evict_hidden % 32) return NOSA_ERR_INVALID_ARG;
  if (c->gather_ctas < 0 || c->gather_ctas > 4096) return NOSA_ERR_INVALID_ARG;
  if (!(c->softmax_scale >= 0.f) || (c->flags & ~(NOSA_F_TEST_ZERO_WAIT | NOSA_F_TEST_BAD_SLOT | NOSA_F_UNFUSED_STEP | NOSA_F_DMA_BIAS |
                                               NOSA_F_TEST_RADIX_TOPK | NOSA_F_TEST_PREFILL_WIDE)))
    return NOSA_ERR_INVALID_ARG;
  if (c->score_ctas < 0 || c->score_ctas > 8) return NOSA_ERR_INVALID_ARG;
  if (c->attend_blocks_per_cta < 0 || c->attend_blocks_per_cta > kMaxBlocksPerCta) return NOSA_ERR_INVALID_ARG;
  if (c->attend_merge < NOSA_MERGE_AUTO || c->attend_merge > NOSA_MERGE_CLUSTER) return NOSA_ERR_INVALID_ARG;
  if (c->decode_cluster < 0 || c->decode_cluster > 8) return NOSA_ERR_INVALID_ARG;
  if (c->decode_teams < 0 || c->decode_teams > 2) return NOSA_ERR_INVALID_ARG;
  if (c->decode_stages != 0 && (c->decode_stages < 2 || c->decode_stages > 6)) return NOSA_ERR_INVALID_ARG;
  if (c->forecast_streams < 0 || c->forecast_streams > 2) return NOSA_ERR_INVALID_ARG;
  const long long U = (long long)c->batch * c->num_kv_heads;
  if (U > 4096) return NOSA_ERR_INVALID_ARG;
  const long long cap = (long long)c->sink_blocks + c->window_tokens / kBlock + c->k_q + c->k_e;
  if (cap < 1 || cap > kMaxCacheSlots) return NOSA_ERR_INVALID_ARG;
  if (c->cache_slots != 0 && (c->cache_slots < cap || c->cache_slots > kMaxCacheSlots)) return NOSA_ERR_INVALID_ARG;
  if ((long long)c->num_layers * U * cap >= (1ll << 31)) return NOSA_ERR_INVALID_ARG;
  return NOSA_OK;
}

nosa_status nosa_query_sizes(const nosa_config* c, nosa_sizes* out) {
  nosa_status st = nosa_validate_config(c);
  if (st != NOSA_OK) return st;
  if (!out) return NOSA_ERR_INVALID_ARG;
  const Derived d = derive(c);
  const uint64_t L = c->num_layers, U = d.U, nc = std::max(d.nc_max, 1);
  out->units_per_layer = d.U;
  out->group = d.G;
  out->cache_slots = d.cs;
  out->select_slots = d.cap;
  out->pad_ = 0;
  out->max_blocks = d.nb_max;
  out->max_windows = d.nc_max;
  out->evict_words = d.ev_words;
  out->host_store_bytes = L * U * d.nb_max * (uint64_t)kBlockBytes;
  const uint64_t per_unit = (uint64_t)d.cs * kBlockBytes + nc * kHeadDim * 2 + 32 * kHeadDim * 2 +
                            (uint64_t)d.nb_max * kBlock * 4 + nc * 4 + (uint64_t)d.nb_max * 12 + d.ev_words * 4ull +
                            (uint64_t)d.cap * 4 * 6 + (uint64_t)d.cs * 4 * 2 + 4 * 4;
  const int score_chunks = cdiv(nc, kWindowsPerCta);
  const uint64_t scratch = U * d.G * nc * 4 + U * score_chunks * kMaxGroup * 8 +
                           U * (uint64_t)d.cap * kMaxGroup * kPartStride * 4 + (3 * U + 1) * 4;
  out->device_state_bytes = L * U * per_unit + L * c->num_kv_heads * (uint64_t)kHeadDim * d.h * 4 + scratch;
  return NOSA_OK;
}

nosa_status nosa_create(const nosa_config* cfg, void* stream, nosa_ctx** out) {
  if (!out) return NOSA_ERR_INVALID_ARG;
  *out = nullptr;
  nosa_status st = nosa_validate_config(cfg);
  if (st != NOSA_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return NOSA_ERR_CUDA;
  }
  nosa_ctx* c = new (std::nothrow) nosa_ctx();
  if (!c) return NOSA_ERR_OOM;
  c->cfg = *cfg;
  nosa_query_sizes(cfg, &c->sz);
  const Derived d = derive(cfg);
  c->L = cfg->num_layers;
  c->B = cfg->batch;
  c->Hq = cfg->num_q_heads;
  c->Hkv = cfg->num_kv_heads;
  c->G = d.G;
  c->d = kHeadDim;
  c->U = d.U;
  c->h = d.h;
  c->nw = d.nw;
  c->cap = d.cap;
  c->cs = d.cs;
  c->stream = (cudaStream_t)stream;
  c->device = dev;
  cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, dev);
  c->T_host.assign(c->L, 0);
  c->sel_T.assign(c->L, -1);
  c->ev_pref.assign(c->L, nullptr);
  c->ev_sel.assign(c->L, nullptr);
  // forecast pipeline: the selections on their own stream (forecast_streams = 1: one prefetch
  // stream for selections and gathers, in order)
  c->forecast_split = cfg->forecast_streams != 1;
  c->pref_pending.assign(c->L, 0);
  c->fetch_T.assign(c->L, -1);

  const size_t LU = (size_t)c->L * c->U;
  const size_t nc = std::max(d.nc_max, 1);
  // selector: one cluster of up to 8 CTAs per unit, each scoring a multiple of 128 windows, and
  // about two CTAs per SM in total: a unit's cluster lives mostly in its leader's serial phase,
  // so at large batch more units in flight beat more CTAs per unit (measured: one CTA per unit
  // at 256 units, four at 64 units with 64K contexts)
  c->score_chunks = std::max(1, std::min({8, cdiv(nc, kWindowsPerCta), 2 * std::max(c->num_sms, 1) / c->U}));
  if (cfg->score_ctas > 0) c->score_chunks = cfg->score_ctas;
  for (;;) {  // more CTAs per unit while one CTA's logits would not fit its shared memory
    c->score_wpc = cdiv(cdiv(nc, c->score_chunks), 16 * kScoreWarps) * 16 * kScoreWarps;
    if (c->score_chunks >= 8 || score_select_smem(layer_state(c, 0)) <= 200 * 1024) break;
    ++c->score_chunks;
  }
  // attend: 8 to 16 selected blocks per CTA, about four CTAs' worth per SM in total (measured
  // best at the batch-128/256 and 64K-context workloads: fewer, longer CTAs starve the host
  // copies of parallelism, more CTAs spend their time in set-up and merging).  The split-K
  // partials are merged by a small merge kernel: merging inside a thread-block cluster per unit
  // (NOSA_MERGE_CLUSTER) makes a cluster's CTAs hold their SMs until the slowest one is done and
  // measured 5-17 % slower at every workload, batch 8 included; merging in the unit's last CTA
  // (NOSA_MERGE_TICKET, the context-free entry point's merge) 1-16 % slower.
  const int sms = std::max(c->num_sms, 1);
  int bpc = cdiv((long long)c->U * d.cap, 4ll * sms);
  bpc = std::min(std::max(bpc, 8), 16);
  if (cfg->attend_blocks_per_cta > 0) bpc = cfg->attend_blocks_per_cta;
  if (init_attend() != cudaSuccess) {  // the cluster query below needs the kernel's smem limit set
    (void)cudaGetLastError();
    delete c;
    return NOSA_ERR_CUDA;
  }
  // internal modes: 0 ticket, 1 cluster, 2 merge kernel
  c->attend_mode = cfg->attend_merge == NOSA_MERGE_TICKET ? 0 : cfg->attend_merge == NOSA_MERGE_CLUSTER ? 1 : 2;
  if (c->attend_mode == 1) {  // the unit's CTAs must form one cluster: widen the chunks until they do
    const int max_cluster = attend_max_cluster();
    while (cdiv(d.cap, bpc) > max_cluster && bpc < kMaxBlocksPerCta) ++bpc;
    if (cdiv(d.cap, bpc) > max_cluster) c->attend_mode = 2;
  }
  c->attend_blocks_per_cta = bpc;
  c->attend_chunks = cdiv(d.cap, bpc);
  c->gather_ctas = cfg->gather_ctas > 0 ? cfg->gather_ctas : (cfg->batch < 32 ? 16 : 32);
  // Fused decode kernel: one cluster of dec_cs CTAs per unit, each CTA dec_teams attention
  // workers of four warps.  It pays off while all units' clusters are resident at once (the
  // small batches where the step is latency bound): the largest cluster of 8 or 4 CTAs for
  // which that holds is taken, else the step runs as three kernels, as it does when the cache
  // has more slots than a CTA has threads.  NOSA_F_UNFUSED_STEP turns it off; decode_cluster,
  // decode_teams and decode_stages override the choices.
  c->dec_cs = 0;
  c->dec_teams = cfg->decode_teams > 0 ? cfg->decode_teams : 2;
  c->dec_nst = cfg->decode_stages > 0 ? cfg->decode_stages : 3;
  if (!(cfg->flags & NOSA_F_UNFUSED_STEP) && d.cs <= 128 * c->dec_teams) {  // a thread per cache slot
    int optin = 0;
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    std::vector<int> sizes = {8, 4};  // with clusters of 2 the selector and attention are too narrow
    const bool force = cfg->decode_cluster > 0;
    if (force) sizes = {cfg->decode_cluster};
    const int warps = 4 * c->dec_teams;
    for (int cs : sizes) {
      c->dec_cs = cs;
      c->dec_wpc = cdiv(cdiv(nc, cs), 16 * warps) * 16 * warps;
      const LayerState sd = decode_state(c, 0);
      const bool ok = decode_smem_bytes(sd, c->dec_teams, c->dec_nst) + 24 * 1024 <= (size_t)optin &&
                      init_decode(sd, c->dec_teams, c->dec_nst) == cudaSuccess;
      const int active = ok ? decode_active_clusters(sd, c->dec_teams, c->dec_nst, cs) : 0;
      (void)cudaGetLastError();
      if (active >= 1 && (force || active >= c->U)) break;
      c->dec_cs = 0;
    }
  }

  // pinned, mapped host store
  const size_t host_bytes = c->sz.host_store_bytes;
  if (cudaHostAlloc((void**)&c->host_kv, host_bytes, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) {
    (void)cudaGetLastError();
    c->host_kv = nullptr;
    free_ctx(c);
    return NOSA_ERR_HOST_ALLOC;
  }
  if (cudaHostGetDevicePointer((void**)&c->host_kv_dev, c->host_kv, 0) != cudaSuccess) {
    (void)cudaGetLastError();
    free_ctx(c);
    return NOSA_ERR_CUDA;
  }
  bool oom = false;
  auto dalloc = [&](auto** p, size_t bytes) {
    if (oom) return;
    if (cudaMalloc((void**)p, std::max<size_t>(bytes, 16)) != cudaSuccess) {
      (void)cudaGetLastError();
      *p = nullptr;
      oom = true;
    }
  };
  dalloc(&c->cache, LU * d.cs * (size_t)kBlockBytes);
  dalloc(&c->kt, LU * nc * kHeadDim * 2);
  dalloc(&c->kring, LU * 32 * kHeadDim * 2);
  dalloc(&c->se_tok, LU * (size_t)d.nb_max * kBlock * 4);
  dalloc(&c->se_win, LU * nc * 4);
  dalloc(&c->se_blk, LU * d.nb_max * 4);
  dalloc(&c->W1, (size_t)c->L * c->Hkv * kHeadDim * d.h * 4);
  dalloc(&c->W2, (size_t)c->L * c->Hkv * d.h * 4);
  dalloc(&c->slot_blk, LU * d.cs * 4);
  dalloc(&c->last_used, LU * d.cs * 4);
  dalloc(&c->blk2slot, LU * d.nb_max * 4);
  dalloc(&c->sel, LU * d.cap * 4);
  dalloc(&c->sel_kind, LU * d.cap * 4);
  dalloc(&c->sel_slot, LU * d.cap * 4);
  dalloc(&c->sel_new, LU * d.cap * 4);
  dalloc(&c->n_sel, LU * 4);
  dalloc(&c->fetch, LU * d.cap * 8);
  dalloc(&c->n_fetch, LU * 4);
  dalloc(&c->gamma, LU * 8);
  dalloc(&c->evicted, LU * d.ev_words * 4);
  dalloc(&c->T, c->L * sizeof(int));
  dalloc(&c->err, sizeof(int));
  dalloc(&c->stats, sizeof(DevStats));
  dalloc(&c->sq_blk, LU * d.nb_max * 4);
  dalloc(&c->apart, (size_t)c->U * c->attend_chunks * kMaxGroup * kPartStride * 4);
  dalloc(&c->tickets, (3 * (size_t)c->U + 1) * 4);
  dalloc(&c->stage_q, (size_t)c->B * c->Hq * kHeadDim * 2);
  dalloc(&c->step_q, (size_t)c->L * c->B * c->Hq * kHeadDim * 2);
  dalloc(&c->step_out, (size_t)c->L * c->B * c->Hq * kHeadDim * 2);
  dalloc(&c->step_k, (size_t)c->L * c->U * kHeadDim * 2);
  dalloc(&c->step_v, (size_t)c->L * c->U * kHeadDim * 2);
  dalloc(&c->stage_out, (size_t)c->B * c->Hq * kHeadDim * 2);
  dalloc(&c->stage_k, (size_t)c->U * kHeadDim * 2);
  dalloc(&c->stage_v, (size_t)c->U * kHeadDim * 2);
  dalloc(&c->bulk_k, (size_t)c->U * c->stage_tok_cap * kHeadDim * 2);
  dalloc(&c->bulk_v, (size_t)c->U * c->stage_tok_cap * kHeadDim * 2);
  if (oom) {
    free_ctx(c);
    return NOSA_ERR_OOM;
  }
  // initial state: empty cache, nothing evicted, pooled eviction scores at -inf
  bool ok = cudaMemset(c->cache, 0, LU * d.cs * (size_t)kBlockBytes) == cudaSuccess;
  ok = ok && cudaMemset(c->kt, 0, LU * nc * kHeadDim * 2) == cudaSuccess;
  ok = ok && cudaMemset(c->kring, 0, LU * 32 * kHeadDim * 2) == cudaSuccess;
  ok = ok && cudaMemset(c->se_tok, 0, LU * (size_t)d.nb_max * kBlock * 4) == cudaSuccess;
  ok = ok && cudaMemset(c->se_win, 0, LU * nc * 4) == cudaSuccess;
  ok = ok && cudaMemset(c->W1, 0, (size_t)c->L * c->Hkv * kHeadDim * d.h * 4) == cudaSuccess;
  ok = ok && cudaMemset(c->W2, 0, (size_t)c->L * c->Hkv * d.h * 4) == cudaSuccess;
  ok = ok && cudaMemset(c->slot_blk, 0xFF, LU * d.cs * 4) == cudaSuccess;
  ok = ok && cudaMemset(c->last_used, 0xFF, LU * d.cs * 4) == cudaSuccess;
  ok = ok && cudaMemset(c->blk2slot, 0xFF, LU * d.nb_max * 4) == cudaSuccess;
  ok = ok && cudaMemset(c->sel, 0xFF, LU * d.cap * 4) == cudaSuccess;
  ok = ok && cudaMemset(c->sel_kind, 0xFF, LU * d.cap * 4) == cudaSuccess;
  ok = ok && cudaMemset(c->sel_slot, 0xFF, LU * d.cap * 4) == cudaSuccess;
  ok = ok && cudaMemset(c->sel_new, 0, LU * d.cap * 4) == cudaSuccess;
  ok = ok && cudaMemset(c->n_sel, 0, LU * 4) == cudaSuccess;
  ok = ok && cudaMemset(c->fetch, 0xFF, LU * d.cap * 8) == cudaSuccess;
  ok = ok && cudaMemset(c->n_fetch, 0, LU * 4) == cudaSuccess;
  ok = ok && cudaMemset(c->gamma, 0, LU * 8) == cudaSuccess;
  ok = ok && cudaMemset(c->evicted, 0, LU * d.ev_words * 4) == cudaSuccess;
  ok = ok && cudaMemset(c->T, 0, c->L * sizeof(int)) == cudaSuccess;
  ok = ok && cudaMemset(c->err, 0, sizeof(int)) == cudaSuccess;
  ok = ok && cudaMemset(c->tickets, 0, (3 * (size_t)c->U + 1) * 4) == cudaSuccess;
  ok = ok && cudaMemset(c->sq_blk, 0, LU * d.nb_max * 4) == cudaSuccess;
  if (ok) {
    fill_f32<<<std::max(1, std::min(cdiv(LU * d.nb_max, 256), 4096)), 256>>>(c->se_blk, LU * d.nb_max, -INFINITY);
    ok = cudaGetLastError() == cudaSuccess;
  }
  DevStats z{};
  z.gamma_min_bits = 0x3F800000u;  // 1.0f
  ok = ok && cudaMemcpy(c->stats, &z, sizeof(z), cudaMemcpyHostToDevice) == cudaSuccess;
  ok = ok && cudaDeviceSynchronize() == cudaSuccess;
  if (!ok) {
    (void)cudaGetLastError();
    free_ctx(c);
    return NOSA_ERR_CUDA;
  }
  // TMA descriptor over the block cache: (d 128, token 64, K/V 2, flat slot L*U*cs), bf16,
  // boxes of 64 dims x 64 tokens x K+V with the 128-byte swizzle
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) {
    free_ctx(c);
    return NOSA_ERR_CUDA;
  }
  cuuint64_t dims[4] = {(cuuint64_t)kHeadDim, (cuuint64_t)kBlock, 2, (cuuint64_t)LU * d.cs};
  cuuint64_t strides[3] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)kBlockElems * 2, (cuuint64_t)kBlockBytes};
  cuuint32_t box[4] = {64, (cuuint32_t)kBlock, 2, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(&c->tmap_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, c->cache, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    free_ctx(c);
    return NOSA_ERR_CUDA;
  }
  {
    const LayerState s0 = layer_state(c, 0);
    if (init_append(s0) != cudaSuccess || init_score_select(s0) != cudaSuccess) {
      (void)cudaGetLastError();
      free_ctx(c);
      return NOSA_ERR_CUDA;
    }
    // sparse prefill: prompts up to max_context, at most the length the walk's block bitmaps cover
    c->pf_max_tokens = std::min(cfg->max_context, prefill_max_tokens());
    if (init_prefill() != cudaSuccess) {
      (void)cudaGetLastError();
      c->pf_max_tokens = 0;
    }
  }
  // forecast pipeline: a selection and a prefetch stream and their events.  Both streams take the
  // device's highest priority: their kernels (the next layer's selection and its host copies) are
  // on the step's critical path, so their CTAs are scheduled ahead of the current layer's
  // remaining attention CTAs as SMs free up.
  int prio_least = 0, prio_greatest = 0;
  if (cudaDeviceGetStreamPriorityRange(&prio_least, &prio_greatest) != cudaSuccess) {
    (void)cudaGetLastError();
    prio_greatest = 0;
  }
  bool ev_ok =
      cudaStreamCreateWithPriority(&c->pref_stream, cudaStreamNonBlocking, prio_greatest) == cudaSuccess &&
      cudaStreamCreateWithPriority(&c->sel_stream, cudaStreamNonBlocking, prio_greatest) == cudaSuccess &&
      cudaEventCreateWithFlags(&c->ev_fork, cudaEventDisableTiming) == cudaSuccess;
  for (int l = 0; l < c->L && ev_ok; ++l)
    ev_ok = cudaEventCreateWithFlags(&c->ev_pref[l], cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&c->ev_sel[l], cudaEventDisableTiming) == cudaSuccess;
  if (!ev_ok) {
    (void)cudaGetLastError();
    free_ctx(c);
    return NOSA_ERR_CUDA;
  }
  *out = c;
  return NOSA_OK;
}

nosa_status nosa_destroy(nosa_ctx* c) {
  if (!c) return NOSA_OK;
  if (c->pref_stream) cudaStreamSynchronize(c->pref_stream);
  if (c->sel_stream) cudaStreamSynchronize(c->sel_stream);
  cudaStreamSynchronize(c->stream);
  (void)cudaGetLastError();
  free_ctx(c);
  return NOSA_OK;
}

nosa_status nosa_set_stream(nosa_ctx* c, void* stream) {
  if (!c) return NOSA_ERR_INVALID_ARG;
  c->stream = (cudaStream_t)stream;
  return NOSA_OK;
}

// A forecast gather started for `layer` on the prefetch stream finishes before the context's
// stream touches that layer's state again (calls may mix the forecast and plain entry points).
static nosa_status join_layer(nosa_ctx* c, int layer) {
  if (c->pref_pending[layer]) {
    CK(cudaStreamWaitEvent(c->stream, c->ev_pref[layer], 0));
    c->pref_pending[layer] = 0;
  }
  return NOSA_OK;
}

// Everything queued on the context's streams (step, forecast selections, forecast gathers) is done.
static nosa_status sync_all(nosa_ctx* c) {
  CK(cudaStreamSynchronize(c->sel_stream));
  CK(cudaStreamSynchronize(c->pref_stream));
  CK(cudaStreamSynchronize(c->stream));
  return NOSA_OK;
}

nosa_status nosa_set_eviction_head(nosa_ctx* c, int layer, const float* W1, const float* W2) {
  nosa_status st = check_ctx(c, layer);
  if (st != NOSA_OK) return st;
  if (!W1 || !W2) return NOSA_ERR_INVALID_ARG;
  const size_t n1 = (size_t)c->Hkv * kHeadDim * c->h, n2 = (size_t)c->Hkv * c->h;
  st = sync_all(c);
  if (st != NOSA_OK) return st;
  CK(cudaMemcpy(c->W1 + layer * n1, W1, n1 * 4, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(c->W2 + layer * n2, W2, n2 * 4, cudaMemcpyHostToDevice));
  return NOSA_OK;
}

nosa_status nosa_append_kv(nosa_ctx* c, int layer, const uint16_t* k, const uint16_t* v, int n, int src_is_host) {
  nosa_status st = check_ctx(c, layer);
  if (st != NOSA_OK) return st;
  if (!k || !v || n < 1) return NOSA_ERR_INVALID_ARG;
  if ((long long)c->T_host[layer] + n > c->cfg.max_context) return NOSA_ERR_CAPACITY;
  st = join_layer(c, layer);
  if (st != NOSA_OK) return st;
  const LayerState s = layer_state(c, layer);
  const size_t row = kHeadDim * 2;
  if (n == 1) {
    const uint16_t *kd = k, *vd = v;
    if (src_is_host) {
      CK(cudaMemcpyAsync(c->stage_k, k, c->U * row, cudaMemcpyHostToDevice, c->stream));
      CK(cudaMemcpyAsync(c->stage_v, v, c->U * row, cudaMemcpyHostToDevice, c->stream));
      kd = c->stage_k;
      vd = c->stage_v;
    }
    CK(launch_append_one(s, kd, vd, true, c->stream));
  } else if (!src_is_host) {
    CK(launch_append_bulk(s, k, v, c->T_host[layer], n, c->stream));
  } else {
    const int chunk = (int)c->stage_tok_cap;
    for (int t0 = 0; t0 < n; t0 += chunk) {
      const int m = std::min(chunk, n - t0);
      CK(cudaMemcpy2DAsync(c->bulk_k, m * row, k + (size_t)t0 * kHeadDim, (size_t)n * row, m * row, c->U,
                           cudaMemcpyHostToDevice, c->stream));
      CK(cudaMemcpy2DAsync(c->bulk_v, m * row, v + (size_t)t0 * kHeadDim, (size_t)n * row, m * row, c->U,
                           cudaMemcpyHostToDevice, c->stream));
      CK(launch_append_bulk(s, c->bulk_k, c->bulk_v, c->T_host[layer] + t0, m, c->stream));
    }
  }
  c->T_host[layer] += n;
  return NOSA_OK;
}

nosa_status nosa_select(nosa_ctx* c, int layer, const uint16_t* q, int32_t* sel_out, int32_t* nfetch_out) {
  nosa_status st = check_ctx(c, layer);
  if (st != NOSA_OK) return st;
  if (!q) return NOSA_ERR_INVALID_ARG;
  if (c->T_host[layer] < 1) return NOSA_ERR_STATE;
  st = join_layer(c, layer);
  if (st != NOSA_OK) return st;
  const LayerState s = layer_state(c, layer);
  CK(launch_score_select(s, q, true, c->stream));
  if (sel_out) {
    copy_i32<<<cdiv((size_t)c->U * c->cap, 256), 256, 0, c->stream>>>(sel_out, s.sel, (size_t)c->U * c->cap);
    CK(cudaGetLastError());
  }
  if (nfetch_out) {
    copy_i32<<<cdiv(c->U, 256), 256, 0, c->stream>>>(nfetch_out, s.n_fetch, (size_t)c->U);
    CK(cudaGetLastError());
  }
  c->sel_T[layer] = c->T_host[layer];
  return NOSA_OK;
}

nosa_status nosa_fetch(nosa_ctx* c, int layer) {
  nosa_status st = check_ctx(c, layer);
  if (st != NOSA_OK) return st;
  const int ahead = c->sel_T[layer] - c->T_host[layer];  // 1 after a forecast selection
  if (ahead != 0 && ahead != 1) return NOSA_ERR_STATE;
  st = join_layer(c, layer);
  if (st != NOSA_OK) return st;
  CK(launch_gather(layer_state(c, layer), c->gather_ctas, c->stream, ahead));
  c->fetch_T[layer] = c->sel_T[layer];
  return NOSA_OK;
}

// Forecast selection of `layer` for its context after the next append, on `stream`.
static nosa_status forecast_select_on(nosa_ctx* c, int layer, const uint16_t* f, cudaStream_t stream) {
  if (c->T_host[layer] < 1) return NOSA_ERR_STATE;
  if (c->T_host[layer] + 1 > c->cfg.max_context) return NOSA_ERR_CAPACITY;
  if (c->sel_T[layer] == c->T_host[layer] + 1) return NOSA_ERR_STATE;  // one forecast per token
  LayerState s = layer_state(c, layer);
  s.G = 1;  // one forecast head per kv head
  CK(launch_score_select(s, f, true, stream, 1));
  c->sel_T[layer] = c->T_host[layer] + 1;
  return NOSA_OK;
}

nosa_status nosa_forecast_select(nosa_ctx* c, int layer, const uint16_t* f) {
  nosa_status st = check_ctx(c, layer);
  if (st != NOSA_OK) return st;
  if (!f) return NOSA_ERR_INVALID_ARG;
  return forecast_select_on(c, layer, f, c->stream);
}

nosa_status nosa_step_forecast(nosa_ctx* c, int layer, const uint16_t* q, const uint16_t* k_new,
                               const uint16_t* v_new, uint16_t* out, const uint16_t* f_next, int next_layer) {
  nosa_status st = check_ctx(c, layer);
  if (st != NOSA_OK) return st;
  if (!q || !k_new || !v_new || !out) return NOSA_ERR_INVALID_ARG;
  if (c->sel_T[layer] != c->T_host[layer] + 1) return NOSA_ERR_STATE;  // no forecast for this token
  if (f_next) {
    if (next_layer < 0 || next_layer >= c->L || next_layer == layer) return NOSA_ERR_INVALID_ARG;
    if (c->sel_T[next_layer] == c->T_host[next_layer] + 1) return NOSA_ERR_STATE;
    if (c->T_host[next_layer] + 1 > c->cfg.max_context) return NOSA_ERR_CAPACITY;
    // the next layer's state was last written by work already queued on the step stream
    // the selection on its own stream, the gather after it on the prefetch stream: the next
    // call's selection (another layer) need not wait for this gather
    cudaStream_t ss = c->forecast_split ? c->sel_stream : c->pref_stream;
    CK(cudaEventRecord(c->ev_fork, c->stream));
    CK(cudaStreamWaitEvent(ss, c->ev_fork, 0));
    st = forecast_select_on(c, next_layer, f_next, ss);
    if (st != NOSA_OK) return st;
    if (c->forecast_split) {
      CK(cudaEventRecord(c->ev_sel[next_layer], c->sel_stream));
      CK(cudaStreamWaitEvent(c->pref_stream, c->ev_sel[next_layer], 0));
    }
    CK(launch_gather(layer_state(c, next_layer), c->gather_ctas, c->pref_stream, 1));
    c->fetch_T[next_layer] = c->sel_T[next_layer];
    CK(cudaEventRecord(c->ev_pref[next_layer], c->pref_stream));
    c->pref_pending[next_layer] = 1;
  }
  if (c->pref_pending[layer]) {
    CK(cudaStreamWaitEvent(c->stream, c->ev_pref[layer], 0));
    c->pref_pending[layer] = 0;
  }
  const LayerState s = layer_state(c, layer);
  CK(launch_append_one(s, k_new, v_new, true, c->stream));
  c->T_host[layer] += 1;
  const int fused = c->fetch_T[layer] != c->T_host[layer];  // no prefetch ran: attend copies itself
  CK(launch_attend(s, &c->tmap_cache, q, out, fused, true, c->stream));
  return NOSA_OK;
}

nosa_status nosa_forecast_join(nosa_ctx* c) {
  if (!c) return NOSA_ERR_INVALID_ARG;
  for (int l = 0; l < c->L; ++l) {
    if (!c->pref_pending[l]) continue;
    CK(cudaStreamWaitEvent(c->stream, c->ev_pref[l], 0));
    c->pref_pending[l] = 0;
  }
  return NOSA_OK;
}

nosa_status nosa_attend(nosa_ctx* c, int layer, const uint16_t* q, uint16_t* out) {
  nosa_status st = check_ctx(c, layer);
  if (st != NOSA_OK) return st;
  if (!q || !out) return NOSA_ERR_INVALID_ARG;
  if (c->sel_T[layer] != c->T_host[layer]) return NOSA_ERR_STATE;
  st = join_layer(c, layer);
  if (st != NOSA_OK) return st;
  // without a nosa_fetch since the selection, the attend CTAs fetch the new blocks themselves
  const int fused = c->fetch_T[layer] != c->T_host[layer];
  CK(launch_attend(layer_state(c, layer), &c->tmap_cache, q, out, fused, true, c->stream));
  return NOSA_OK;
}

nosa_status nosa_step(nosa_ctx* c, int layer, const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                      uint16_t* out) {
  nosa_status st = check_ctx(c, layer);
  if (st != NOSA_OK) return st;
  if (!q || !k_new || !v_new || !out) return NOSA_ERR_INVALID_ARG;
  if (c->T_host[layer] + 1 > c->cfg.max_context) return NOSA_ERR_CAPACITY;
  st = join_layer(c, layer);
  if (st != NOSA_OK) return st;
  if (c->dec_cs > 0) {  // one fused kernel
    CK(launch_decode(decode_state(c, layer), &c->tmap_cache, q, k_new, v_new, out, c->dec_teams, c->dec_nst, true,
                     c->stream));
  } else {
    const LayerState s = layer_state(c, layer);
    CK(launch_score_select(s, q, true, c->stream, 0, k_new, v_new));  // appends the token first
    CK(launch_attend(s, &c->tmap_cache, q, out, 1, true, c->stream));  // the fetch runs inside attend
  }
  c->T_host[layer] += 1;
  c->sel_T[layer] = c->T_host[layer];
  return NOSA_OK;
}

// The device address of page-locked host memory (cudaHostAlloc / cudaHostRegister), or
// nullptr for memory the device cannot address (pageable allocations).
static void* pinned_device_view(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

nosa_status nosa_step_host(nosa_ctx* c, int layer, const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                           uint16_t* out) {
  nosa_status st = check_ctx(c, layer);
  if (st != NOSA_OK) return st;
  if (!q || !k_new || !v_new || !out) return NOSA_ERR_INVALID_ARG;
  // Page-locked buffers are read and written by the kernels in place over the host link:
  // no copy operations between the three kernels, so they stay chained.
  void *dq = pinned_device_view(q), *dk = pinned_device_view(k_new), *dv = pinned_device_view(v_new),
       *dout = pinned_device_view(out);
  if (dq && dk && dv && dout)
    return nosa_step(c, layer, static_cast<const uint16_t*>(dq), static_cast<const uint16_t*>(dk),
                     static_cast<const uint16_t*>(dv), static_cast<uint16_t*>(dout));
  const size_t qbytes = (size_t)c->B * c->Hq * kHeadDim * 2, kvbytes = (size_t)c->U * kHeadDim * 2;
  CK(cudaMemcpyAsync(c->stage_q, q, qbytes, cudaMemcpyHostToDevice, c->stream));
  CK(cudaMemcpyAsync(c->stage_k, k_new, kvbytes, cudaMemcpyHostToDevice, c->stream));
  CK(cudaMemcpyAsync(c->stage_v, v_new, kvbytes, cudaMemcpyHostToDevice, c->stream));
  st = nosa_step(c, layer, c->stage_q, c->stage_k, c->stage_v, c->stage_out);
  if (st != NOSA_OK) return st;
  CK(cudaMemcpyAsync(out, c->stage_out, qbytes, cudaMemcpyDeviceToHost, c->stream));
  return NOSA_OK;
}

nosa_status nosa_step_host_all(nosa_ctx* c, const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                               uint16_t* out) {
  if (!c || !q || !k_new || !v_new || !out) return NOSA_ERR_INVALID_ARG;
  for (int l = 0; l < c->L; ++l) {  // everything nosa_step checks, for every layer, before anything runs
    const nosa_status st = check_ctx(c, l);
    if (st != NOSA_OK) return st;
    if (c->T_host[l] + 1 > c->cfg.max_context) return NOSA_ERR_CAPACITY;
  }
  const size_t qL = (size_t)c->B * c->Hq * kHeadDim, kvL = (size_t)c->U * kHeadDim;  // elements per layer
  CK(cudaMemcpyAsync(c->step_q, q, c->L * qL * 2, cudaMemcpyHostToDevice, c->stream));
  CK(cudaMemcpyAsync(c->step_k, k_new, c->L * kvL * 2, cudaMemcpyHostToDevice, c->stream));
  CK(cudaMemcpyAsync(c->step_v, v_new, c->L * kvL * 2, cudaMemcpyHostToDevice, c->stream));
  for (int l = 0; l < c->L; ++l) {
    const nosa_status st = nosa_step(c, l, c->step_q + l * qL, c->step_k + l * kvL, c->step_v + l * kvL,
                                     c->step_out + l * qL);
    if (st != NOSA_OK) return st;
  }
  CK(cudaMemcpyAsync(out, c->step_out, c->L * qL * 2, cudaMemcpyDeviceToHost, c->stream));
  return NOSA_OK;
}

// [2][U][n][ceil(nb / 32)] bitmap words over the prompt's nb blocks: each position's query-aware,
// then query-agnostic picks
static size_t prefill_pick_bytes(const nosa_ctx* c, int n_tokens) {
  return (size_t)c->U * (size_t)n_tokens * (size_t)cdiv(cdiv(n_tokens, kBlock), 32) * sizeof(uint32_t);
}

size_t nosa_prefill_scratch_bytes(nosa_ctx* c, int n_tokens) {
  if (!c || n_tokens < 1) return 0;
  return 2 * prefill_pick_bytes(c, n_tokens);
}

nosa_status nosa_prefill(nosa_ctx* c, int layer, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         int n_tokens, uint16_t* out, void* scratch, size_t scratch_bytes) {
  nosa_status st = check_ctx(c, layer);
  if (st != NOSA_OK) return st;
  if (!q || !k || !v || !out || !scratch || n_tokens < 1) return NOSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) % 16) return NOSA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(q) % 16 || reinterpret_cast<uintptr_t>(scratch) % 16) return NOSA_ERR_INVALID_ARG;
  if (c->T_host[layer] != 0) return NOSA_ERR_STATE;  // a prefill starts an empty layer
  if (n_tokens > c->cfg.max_context || n_tokens > c->pf_max_tokens) return NOSA_ERR_CAPACITY;
  if (scratch_bytes < nosa_prefill_scratch_bytes(c, n_tokens)) return NOSA_ERR_CAPACITY;
  st = join_layer(c, layer);
  if (st != NOSA_OK) return st;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return NOSA_ERR_CUDA;
  // the prompt's K and V, [U][n][d] each: boxes of 64 dims x 64 tokens with the 128-byte swizzle
  CUtensorMap tk, tv;
  cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)n_tokens, (cuuint64_t)c->U};
  cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)n_tokens * kHeadDim * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)kBlock, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  for (int i = 0; i < 2; ++i)
    if (enc(i ? &tv : &tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(i ? v : k), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return NOSA_ERR_INVALID_ARG;
  const LayerState s = layer_state(c, layer);
  // the layer's compressed keys [U][nc_max][d]: boxes of 64 dims x 128 windows
  CUtensorMap tkt;
  {
    cuuint64_t kdims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)s.nc_max, (cuuint64_t)c->U};
    cuuint64_t kstr[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)s.nc_max * kHeadDim * 2};
    cuuint32_t kbox[3] = {64, 128, 1};
    if (enc(&tkt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, s.kt, kdims, kstr, kbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return NOSA_ERR_INVALID_ARG;
  }
  CK(launch_append_bulk(s, k, v, 0, n_tokens, c->stream));
  uint32_t* qsel = static_cast<uint32_t*>(scratch);
  uint32_t* esel = reinterpret_cast<uint32_t*>(static_cast<unsigned char*>(scratch) + prefill_pick_bytes(c, n_tokens));
  CK(launch_prefill(s, &tk, &tv, &tkt, q, k, v, out, qsel, esel, n_tokens,
                    (c->cfg.flags & NOSA_F_TEST_PREFILL_WIDE) != 0, c->stream));
  c->T_host[layer] = n_tokens;
  c->sel_T[layer] = n_tokens;
  c->fetch_T[layer] = n_tokens;  // every cache slot holds its block
  return NOSA_OK;
}

nosa_status nosa_step_plan(nosa_ctx* c, int32_t* kernels_per_layer, int32_t* cluster_size) {
  if (!c) return NOSA_ERR_INVALID_ARG;
  // fused: one kernel; else the selector (which appends) and the attention, plus the merge kernel
  if (kernels_per_layer) *kernels_per_layer = c->dec_cs > 0 ? 1 : (c->attend_mode == 2 ? 3 : 2);
  if (cluster_size) *cluster_size = c->dec_cs;
  return NOSA_OK;
}

nosa_status nosa_sync(nosa_ctx* c) {
  if (!c) return NOSA_ERR_INVALID_ARG;
  const nosa_status ss = sync_all(c);
  if (ss != NOSA_OK) return ss;
  int e = 0;
  CK(cudaMemcpy(&e, c->err, sizeof(int), cudaMemcpyDeviceToHost));
  std::vector<int> T(c->L);
  CK(cudaMemcpy(T.data(), c->T, c->L * sizeof(int), cudaMemcpyDeviceToHost));
  for (int l = 0; l < c->L; ++l) {  // graph replays advance the device lengths only
    if (T[l] != c->T_host[l]) {   // keep the selection (and fetch) a forecast ahead, or not, as captured
      const int ds = c->sel_T[l] - c->T_host[l], df = c->fetch_T[l] - c->T_host[l];
      if (ds == 0 || ds == 1) c->sel_T[l] = T[l] + ds;
      if (df == 0 || df == 1) c->fetch_T[l] = T[l] + df;
    }
    c->T_host[l] = T[l];
  }
  if (e && !c->failed) c->failed = err_to_status(e);
  return c->failed ? (nosa_status)c->failed : NOSA_OK;
}

nosa_status nosa_reset_state(nosa_ctx* c) {
  if (!c) return NOSA_ERR_INVALID_ARG;
  const nosa_status ss = sync_all(c);
  if (ss != NOSA_OK) return ss;
  CK(cudaMemset(c->err, 0, sizeof(int)));
  c->failed = 0;
  return NOSA_OK;
}

nosa_status nosa_context_length(nosa_ctx* c, int layer, int32_t* T_out) {
  if (!c || !T_out || layer < 0 || layer >= c->L) return NOSA_ERR_INVALID_ARG;
  nosa_status st = nosa_sync(c);
  *T_out = c->T_host[layer];
  return st;
}

nosa_status nosa_get_stats(nosa_ctx* c, nosa_stats* out) {
  if (!c || !out) return NOSA_ERR_INVALID_ARG;
  const nosa_status ss = sync_all(c);
  if (ss != NOSA_OK) return ss;
  DevStats d;
  CK(cudaMemcpy(&d, c->stats, sizeof(d), cudaMemcpyDeviceToHost));
  out->selections = d.selections;
  out->gamma_samples = d.gamma_samples;
  out->gamma_mean = d.gamma_den ? (double)d.gamma_num / (double)d.gamma_den : 1.0;
  float gm;
  memcpy(&gm, &d.gamma_min_bits, 4);
  out->gamma_min = gm;
  out->blocks_fetched = d.blocks_fetched;
  out->bytes_fetched = d.blocks_fetched * (uint64_t)kBlockBytes;
  out->short_selections = d.short_selections;
  return NOSA_OK;
}

nosa_status nosa_reset_stats(nosa_ctx* c) {
  if (!c) return NOSA_ERR_INVALID_ARG;
  const nosa_status ss = sync_all(c);
  if (ss != NOSA_OK) return ss;
  DevStats z{};
  z.gamma_min_bits = 0x3F800000u;
  CK(cudaMemcpy(c->stats, &z, sizeof(z), cudaMemcpyHostToDevice));
  return NOSA_OK;
}

nosa_status nosa_debug_scores(nosa_ctx* c, int layer, float* sq, float* se) {
  if (!c || layer < 0 || layer >= c->L) return NOSA_ERR_INVALID_ARG;
  const nosa_status ss = sync_all(c);
  if (ss != NOSA_OK) return ss;
  const LayerState s = layer_state(c, layer);
  const size_t n = (size_t)c->U * s.nb_max * 4;
  if (sq) CK(cudaMemcpy(sq, s.sq_blk, n, cudaMemcpyDeviceToHost));
  if (se) CK(cudaMemcpy(se, s.se_blk, n, cudaMemcpyDeviceToHost));
  return NOSA_OK;
}

nosa_status nosa_export_state(nosa_ctx* c, int layer, const nosa_state_view* v) {
  if (!c || !v || layer < 0 || layer >= c->L) return NOSA_ERR_INVALID_ARG;
  const nosa_status ss = sync_all(c);
  if (ss != NOSA_OK) return ss;
  const LayerState s = layer_state(c, layer);
  const size_t U = c->U, cap = c->cap, cs = c->cs;
  auto cp = [&](void* dst, const void* src, size_t bytes) {
    return dst ? cudaMemcpy(dst, src, bytes, cudaMemcpyDeviceToHost) : cudaSuccess;
  };
  CK(cp(v->sel, s.sel, U * cap * 4));
  CK(cp(v->sel_kind, s.sel_kind, U * cap * 4));
  CK(cp(v->sel_slot, s.sel_slot, U * cap * 4));
  CK(cp(v->n_sel, s.n_sel, U * 4));
  CK(cp(v->fetch, s.fetch, U * cap * 8));
  CK(cp(v->n_fetch, s.n_fetch, U * 4));
  CK(cp(v->slot_blk, s.slot_blk, U * cs * 4));
  CK(cp(v->last_used, s.last_used, U * cs * 4));
  CK(cp(v->evicted, s.evicted, U * s.ev_words * 4));
  CK(cp(v->kt, s.kt, U * s.nc_max * kHeadDim * 2));
  CK(cp(v->se_win, s.se_win, U * s.nc_max * 4));
  CK(cp(v->se_blk, s.se_blk, U * s.nb_max * 4));
  CK(cp(v->gamma, s.gamma, U * 8));
  return NOSA_OK;
}

}  // extern "C"
