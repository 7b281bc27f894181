// Host-side declarations of libnosa.so: the context object behind nosa_ctx* and the
// launchers and set-up functions each kernel translation unit exports.
#pragma once

#include "nosa_internal.cuh"

struct nosa_ctx {
  nosa_config cfg;
  nosa_sizes sz;
  int L, B, Hq, Hkv, G, d, U, h, nw, cap, cs;  // cap: blocks of a selection; cs: cache slots per unit
  cudaStream_t stream;
  int device;
  int num_sms;
  // pinned host store and its device alias
  uint16_t* host_kv;
  uint16_t* host_kv_dev;
  size_t host_layer_elems;
  // device state (all layers, one allocation each)
  uint16_t *cache, *kt, *kring;
  float *se_tok, *se_win, *se_blk, *W1, *W2;
  int32_t *slot_blk, *last_used, *blk2slot, *sel, *sel_kind, *sel_slot, *sel_new, *n_sel, *fetch, *n_fetch, *gamma;
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
  // sparse prefill: the longest prompt (0: the prefill kernels could not be set up)
  int pf_max_tokens;
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
  cudaStream_t pref_stream;  // the forecast gathers
  cudaStream_t sel_stream;   // the forecast selections (a layer's overlaps the previous layer's gather)
  int forecast_split;        // 1: selections on sel_stream; 0: selections and gathers in order on pref_stream
  cudaEvent_t ev_fork;
  std::vector<cudaEvent_t> ev_pref;  // per layer: its forecast gather is done
  std::vector<cudaEvent_t> ev_sel;   // per layer: its forecast selection is done
  std::vector<char> pref_pending;
};

namespace nosa {
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
// sparse prefill of an empty layer (after the bulk append of the prompt): every position's
// query-aware picks into qsel, then its query-agnostic picks in order into esel (both [U][n]
// [ceil(nb / 32)] bitmap words over the prompt's nb blocks), cache slots refreshed from the
// prompt, attention of every position
cudaError_t init_prefill();
int prefill_max_tokens();
// tk, tv: the prompt's K and V; tkt: the layer's compressed keys [U][nc_max][d] (boxes of 64 dims x
// 128 windows, 128-byte swizzle)
cudaError_t launch_prefill(const LayerState& s, const CUtensorMap* tk, const CUtensorMap* tv, const CUtensorMap* tkt,
                           const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* out, uint32_t* qsel,
                           uint32_t* esel, int n, bool wide, cudaStream_t st);  // wide: the long-prompt walk at any length
}  // namespace nosa
