// a2-a4 phases of the scorer and the two-part selector, shared by the selector
// kernel and the fused decode kernel.
//
// One thread-block cluster per unit, 128 or 256 threads per CTA (the leader's
// slot scan takes one thread per cache slot): CTA r of the cluster scores
// compressed windows [r*wpc, (r+1)*wpc), wpc a multiple of 16 * warps.
//   1. z_{h,i} = q_h . K~_i * scale on the tensor cores (mma.sync m16n8k16,
//      16 windows as M, the GQA group's heads as N = 8), kept in shared memory,
//      with this CTA's per-head softmax statistics (max, sum of exp).
//   2. cluster barrier; every CTA reads all CTAs' statistics through
//      distributed shared memory, forms the group softmax over all windows
//      summed over the heads (SparDA summary, "lightweight design": the block
//      selector aggregates the group's heads through a softmax) and max-pools
//      its windows onto the 64-token blocks they overlap (NOSA explainer
//      eq. 5-6), combining into the leader CTA's block scores with remote
//      atomic max.
//   3. every CTA ranks the candidate blocks it owns and sends its k_q best to
//      the leader; after a third barrier the leader selects: the top-k_q of
//      those query-aware candidates, then
//      k_e blocks by the pooled eviction score among candidates never dropped
//      before (wiki "How NOSA works": query-aware picks set to +inf, the rest
//      filled by the query-agnostic score, never-reselect constraint); sink and
//      window blocks; sticky eviction update; set difference against the block
//      cache with ascending free-slot assignment (wiki "NOSI": set-difference
//      kernel, only changed blocks are swapped); fetch list.
// The leader's inputs for step 3 (pooled s^e, slot tables, eviction bitmap) are
// requested before step 1 and arrive while it runs.
#pragma once

#include <cooperative_groups.h>

#include "nosa_internal.cuh"
#include "ptx.cuh"

namespace nosa {

namespace selcore {

namespace cg = cooperative_groups;

constexpr uint8_t F_CAND = 1, F_ELIG = 2, F_Q = 4, F_E = 8, F_S = 16, F_NEW = 32;
constexpr int kMaxScoreCluster = 8;
constexpr int kSortRankMin = 64;  // owned candidates above which the local ranking sorts (k_q <= 32)

struct SelShared {
  int cand_n[kMaxScoreCluster];  // leader: local winners per cluster CTA
  int scan[32];
  int hist[256];
  int free_by_rank[256];
  float cmax[kScoreWarps][kMaxGroup];
  float Mloc[kMaxGroup], Sloc[kMaxGroup];  // this CTA's softmax statistics (read remotely)
  float Mh[kMaxGroup], invS[kMaxGroup];    // the unit's statistics
  int4 wsum[kScoreWarps];
  int cofs[kMaxScoreCluster + 1];
  float zx[kMaxGroup];  // logits of the window just before this CTA's range (pooled here too)
  float sqx;            // its query-aware score
  int lumax[kMaxCacheSlots / 32];     // per warp: the latest selection any cache slot served
  uint32_t okey[kMaxCacheSlots];      // cache slots open to new blocks: (last selected + 1, slot)
};

// Composite ranking key: higher score first, then lower block.  Distinct blocks give
// distinct keys, so a rank is one branch-free count of larger keys.
__device__ __forceinline__ unsigned long long rank_key(uint32_t score_key, int blk) {
  return ((unsigned long long)score_key << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)blk);
}

// Rank of key ki among list[0..n): the number of larger keys (loads pipelined, no branches).
__device__ __forceinline__ int count_larger(const unsigned long long* list, int n, unsigned long long ki) {
  int r = 0;
#pragma unroll 8
  for (int j = 0; j < n; ++j) r += list[j] > ki ? 1 : 0;
  return r;
}


// Top-k over the blocks whose flag has `valid` set, run by one warp: sets `mark`
// on the k largest keys, ties to the lower block index.  Radix select on the
// keys' offsets from the smallest valid key, 8-bit digits taken from the
// highest bit of (max - min) down, so the digits spread over the actual range
// of the scores (pooled scores share their high bits) and the shared-memory
// histogram atomics rarely collide; the bins are scanned with warp shuffles.  The keys
// equal to the k-th largest are then taken in ascending block order by ballot.
static __device__ void warp_topk(const uint32_t* keys, uint8_t* flags, int n, int k, uint8_t valid, uint8_t mark,
                          int* hist) {
  const int lane = threadIdx.x & 31;
  if (k <= 0) return;
  int cnt = 0;
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  for (int b = lane; b < n; b += 32)
    if (flags[b] & valid) {
      ++cnt;
      kmin = min(kmin, keys[b]);
      kmax = max(kmax, keys[b]);
    }
  cnt = warp_sum(cnt);
  if (cnt <= k) {
    for (int b = lane; b < n; b += 32)
      if (flags[b] & valid) flags[b] |= mark;
    __syncwarp();
    return;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  const int bits = 32 - __clz(kmax - kmin);  // offsets lie in [0, 2^bits)
  uint32_t prefix = 0, pmask = 0;            // over offsets
  int need = k;
  // digits of 8 bits from the top of the offset range down; the last one may be narrower
  for (int top = bits; top > 0; top -= 8) {
    const int shift = max(top - 8, 0);
    const uint32_t dmask = (1u << (top - shift)) - 1u;
    for (int i = lane; i < 256; i += 32) hist[i] = 0;
    __syncwarp();
    for (int b = lane; b < n; b += 32) {
      const uint32_t off = keys[b] - kmin;
      if ((flags[b] & valid) && (off & pmask) == prefix) atomicAdd(&hist[(off >> shift) & dmask], 1);
    }
    __syncwarp();
    int c[8], tot = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // lane owns 8 bins counted down from the top digit
      c[j] = hist[255 - (8 * lane + j)];
      tot += c[j];
    }
    int incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - tot, fd = -1, fa = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (fd < 0 && run < need && run + c[j] >= need) {
        fd = 255 - (8 * lane + j);
        fa = run;
      }
      run += c[j];
    }
    const unsigned int m = __ballot_sync(0xffffffffu, fd >= 0);
    const int src = __ffs(m) - 1;
    const int digit = __shfl_sync(0xffffffffu, fd, src);
    need -= __shfl_sync(0xffffffffu, fa, src);
    prefix |= (uint32_t)digit << shift;
    pmask |= dmask << shift;
    __syncwarp();
  }
  // kmin + prefix is the k-th largest key; `need` keys equal to it are taken, lowest blocks first
  const uint32_t thr = kmin + prefix;
  int taken = 0;
  for (int base = 0; base < n; base += 32) {
    const int b = base + lane;
    const bool v = b < n && (flags[b] & valid);
    const uint32_t key = v ? keys[b] : 0u;
    const bool tie = v && key == thr;
    const unsigned int tm = __ballot_sync(0xffffffffu, tie);
    const int rank = taken + __popc(tm & ((1u << lane) - 1u));
    if ((v && key > thr) || (tie && rank < need)) flags[b] |= mark;
    taken += __popc(tm);
  }
  __syncwarp();
}


// Bitonic sort of one 64-bit key per lane, descending across the warp (15 compare-exchange
// stages through warp shuffles).
__device__ __forceinline__ unsigned long long warp_sort_desc(unsigned long long x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, j);
      // runs of length k alternate direction; the last run (k = 32) is descending
      const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
      x = keep_max ? (x > y ? x : y) : (x < y ? x : y);
    }
  }
  return x;
}

// The 32 largest keys of two descending warp lists, descending: the elementwise maximum of one
// list and the other reversed is a bitonic sequence holding them, which five half-cleaner stages
// sort.
__device__ __forceinline__ unsigned long long warp_merge_top(unsigned long long a, unsigned long long b) {
  const int lane = threadIdx.x & 31;
  const unsigned long long br = __shfl_sync(0xffffffffu, b, 31 - lane);
  unsigned long long x = a > br ? a : br;
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, j);
    x = (lane & j) == 0 ? (x > y ? x : y) : (x < y ? x : y);
  }
  return x;
}


// Floats of the first shared-memory region: the window logits, later reused for
// 64-bit ranking keys (up to 8 * k_q gathered winners, or one per block).
__host__ __device__ inline int zs_floats(const LayerState& s) {
  const int keys64 = 2 * (kMaxScoreCluster * s.k_q > s.nb_max ? kMaxScoreCluster * s.k_q : s.nb_max);
  return kMaxGroup * s.score_wpc > keys64 ? kMaxGroup * s.score_wpc : keys64;
}

// Bytes of dynamic shared memory the phases use: z[kMaxGroup][wpc] and sq[wpc] floats
// (every CTA), then for the leader keys, pooled s^e and the block -> slot map
// [nb_max] each, eviction words, the gathered local winners [8][k_q] (keys and
// blocks), eligible blocks [nb_max], the cache slots' last selections [cslots] and
// flags [nb_max].
__host__ __device__ inline size_t region_bytes(const LayerState& s) {
  return sizeof(float) * ((size_t)zs_floats(s) + s.score_wpc) + 4 * sizeof(uint32_t) * s.nb_max +
         sizeof(uint32_t) * s.ev_words + 2 * sizeof(uint32_t) * kMaxScoreCluster * s.k_q +
         sizeof(int32_t) * s.cslots + s.nb_max + 16;
}

struct Smem {
  float* zs;           // [kMaxGroup][wpc], later ranking keys
  float* sqs;          // [wpc]
  uint32_t* keys;      // leader: [nb_max] pooled query-aware scores (orderable)
  float* sek;          // leader: [nb_max] pooled s^e
  int32_t* b2s;        // leader: [nb_max] block -> slot
  uint32_t* evw;       // leader: [ev_words]
  uint32_t* cand_key;  // leader: [8][k_q] local winners' keys
  int32_t* cand_blk;   // leader: [8][k_q]
  int32_t* lu;         // leader: [cslots] context length of the last selection each slot served
  uint8_t* flags;      // leader: [nb_max]
};

__device__ __forceinline__ Smem layout(unsigned char* dsm, const LayerState& s) {
  Smem m;
  m.zs = reinterpret_cast<float*>(dsm);
  m.sqs = m.zs + zs_floats(s);
  m.keys = reinterpret_cast<uint32_t*>(m.sqs + s.score_wpc);
  m.sek = reinterpret_cast<float*>(m.keys + s.nb_max);
  m.b2s = reinterpret_cast<int32_t*>(m.sek + s.nb_max);
  m.evw = reinterpret_cast<uint32_t*>(m.b2s + s.nb_max);
  m.cand_key = m.evw + s.ev_words;
  m.cand_blk = reinterpret_cast<int32_t*>(m.cand_key + kMaxScoreCluster * s.k_q);
  int32_t* eblk = m.cand_blk + kMaxScoreCluster * s.k_q;  // [nb_max] (reserved)
  m.lu = eblk + s.nb_max;
  m.flags = reinterpret_cast<uint8_t*>(m.lu + s.cslots);
  return m;
}

// A selection's consumer that takes nothing (the selection goes to global memory only).
struct NoDeal {
  __device__ __forceinline__ void operator()(int, int, int, bool, int, int) const {}
};

// q fragments for the scorer.  The k order in each 32-dim chunk is permuted
// identically for A (K~ rows) and B (q), so a thread loads 16 contiguous bytes
// per row and a warp load covers whole sectors.
__device__ __forceinline__ void load_q(uint4 (&qf)[4], const uint16_t* q, int u, int G) {
  const int lane = threadIdx.x & 31, gr = lane >> 2, t4 = lane & 3;
  const uint16_t* qh = q + ((size_t)u * G + min(gr, G - 1)) * kHeadDim;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    qf[c] = gr < G ? *reinterpret_cast<const uint4*>(qh + 32 * c + 8 * t4) : make_uint4(0, 0, 0, 0);
}

// Leader only, before phase 1: request the selection's inputs as asynchronous copies
// into shared memory (waited for with cp_async_wait_all before leader_select).
// Pooled s^e is read for blocks below nb_se only.
// Returns this thread's cache slot's block (thread index < cslots), or -1.
__device__ __forceinline__ int leader_prefetch(const LayerState& s, int u, int nb, int nb_se, const Smem& m) {
  const int tid = threadIdx.x;
  float* sek = m.sek;
  int32_t* b2s = m.b2s;
  uint32_t* evw = m.evw;
  // a selecting CTA requests the selection's inputs now as asynchronous copies into
  // shared memory; they land while the scoring runs (waited for before the selection)
  const float* seg = s.se_blk + (size_t)u * s.nb_max;
  const int32_t* b2g = s.blk2slot + (size_t)u * s.nb_max;
  const uint32_t* evg = s.evicted + (size_t)u * s.ev_words;
  for (int b = tid; b < nb; b += blockDim.x) {
    if (b >= nb_se) {
      cp_async_4(smem_u32(b2s + b), b2g + b);
      continue;
    }
    cp_async_4(smem_u32(sek + b), seg + b);
    cp_async_4(smem_u32(b2s + b), b2g + b);
  }
  for (int w = tid; w < (nb + 31) / 32; w += blockDim.x) cp_async_4(smem_u32(evw + w), evg + w);
  const int32_t* lug = s.last_used + (size_t)u * s.cslots;
  for (int sl = tid; sl < s.cslots; sl += blockDim.x) cp_async_4(smem_u32(m.lu + sl), lug + sl);
  cp_async_commit();
  return tid < s.cslots ? s.slot_blk[(size_t)u * s.cslots + tid] : -1;
}

// Phase 1: this CTA's window logits z (shared memory) and per-head statistics.  Each
// warp issues the key loads of kScoreBatch 16-window tiles together.
template <int kScoreBatch>
__device__ __forceinline__ void score_windows(const LayerState& s, int u, int nc, int rank, const Smem& m,
                                              SelShared& sh, const uint4 (&qf)[4]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gr = lane >> 2, t4 = lane & 3;
  const int G = s.G, wpc = s.score_wpc;
  const int i0 = rank * wpc;
  float* zs = m.zs;
  // ---------------- 1. z for this CTA's windows, per-head max
  const float scale = s.scale;
  float mx[2] = {-INFINITY, -INFINITY};
  // The window just before this CTA's range overlaps this CTA's first block: warp 0 scores it
  // too (the 16-window tile ending with it; its loads go out with the first batch).
  const bool has_x = i0 >= 1 && i0 - 1 < nc;
  uint4 ax[2][4];
  if (warp == 0) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = i0 - 16 + gr + 8 * hr;
      const bool ok = has_x && r >= 0 && r < nc;
      const uint16_t* kr = s.kt + ((size_t)u * s.nc_max + (ok ? r : 0)) * kHeadDim;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        ax[hr][c] = ok ? *reinterpret_cast<const uint4*>(kr + 32 * c + 8 * t4) : make_uint4(0, 0, 0, 0);
    }
  }
  const int nwarps = blockDim.x >> 5;
  const int tiles = wpc / (16 * nwarps);
  for (int t0 = 0; t0 < tiles; t0 += kScoreBatch) {  // the loads of kScoreBatch tiles in flight together
    uint4 a[kScoreBatch][2][4];
#pragma unroll
    for (int tl = 0; tl < kScoreBatch; ++tl)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int r = i0 + (warp * tiles + t0 + tl) * 16 + gr + 8 * hr;
        const bool ok = t0 + tl < tiles && r < nc;
        const uint16_t* kr = s.kt + ((size_t)u * s.nc_max + (ok ? r : 0)) * kHeadDim;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          a[tl][hr][c] = ok ? *reinterpret_cast<const uint4*>(kr + 32 * c + 8 * t4) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
    for (int tl = 0; tl < kScoreBatch; ++tl) {
      if (t0 + tl >= tiles) break;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t* r0 = reinterpret_cast<const uint32_t*>(&a[tl][0][c]);
        const uint32_t* r1 = reinterpret_cast<const uint32_t*>(&a[tl][1][c]);
        const uint32_t* qq = reinterpret_cast<const uint32_t*>(&qf[c]);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint32_t af[4] = {r0[2 * hh], r1[2 * hh], r0[2 * hh + 1], r1[2 * hh + 1]};
          mma_16816(acc, af, qq[2 * hh], qq[2 * hh + 1]);
        }
      }
      const int wl0 = (warp * tiles + t0 + tl) * 16 + gr;  // local window of acc[0..1]
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int wl = wl0 + 8 * (j >> 1), h = 2 * t4 + (j & 1);
        const float z = (i0 + wl < nc) ? acc[j] * scale : -INFINITY;
        zs[h * wpc + wl] = z;
        mx[j & 1] = fmaxf(mx[j & 1], z);
      }
    }
  }
  if (warp == 0) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t* r0 = reinterpret_cast<const uint32_t*>(&ax[0][c]);
      const uint32_t* r1 = reinterpret_cast<const uint32_t*>(&ax[1][c]);
      const uint32_t* qq = reinterpret_cast<const uint32_t*>(&qf[c]);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t af[4] = {r0[2 * hh], r1[2 * hh], r0[2 * hh + 1], r1[2 * hh + 1]};
        mma_16816(acc, af, qq[2 * hh], qq[2 * hh + 1]);
      }
    }
    if (gr == 7) {  // row 15 of the tile: window i0 - 1
      sh.zx[2 * t4] = has_x ? acc[2] * scale : -INFINITY;
      sh.zx[2 * t4 + 1] = has_x ? acc[3] * scale : -INFINITY;
    }
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 4));
    mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 8));
    mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 16));
  }
  if (gr == 0) {
    sh.cmax[warp][2 * t4] = mx[0];
    sh.cmax[warp][2 * t4 + 1] = mx[1];
  }
  __syncthreads();
  if (tid < kMaxGroup) {
    float m = -INFINITY;
    for (int w = 0; w < nwarps; ++w) m = fmaxf(m, sh.cmax[w][tid]);
    sh.Mloc[tid] = m;
  }
  __syncthreads();
  // sum of exp per head over this CTA's windows: warp w handles heads w, w + nwarps, ...
  for (int h = warp; h < G; h += nwarps) {
    const float M = sh.Mloc[h];
    float e = 0.f;
    if (M > -INFINITY)
      for (int wl = lane; wl < wpc; wl += 32) e += expf(zs[h * wpc + wl] - M);  // exp(-inf) = 0
    e = warp_sum(e);
    if (lane == 0) sh.Sloc[h] = e;
  }
}

// Block ownership for pooling and local ranking: block b belongs to the CTA scoring
// window 4b (the first window starting in it), so every window overlapping b
// (4b-1 .. 4b+3) was scored there (window 4b-1 of the first owned block as the extra
// one); the last CTA also takes the blocks that no window starts in.
__device__ __forceinline__ void owned_blocks(const LayerState& s, int nb, int rank, int CS, int& b0, int& b1) {
  const int i0 = rank * s.score_wpc;
  b0 = min(i0 / 4, nb);
  b1 = rank == CS - 1 ? nb : min((i0 + s.score_wpc) / 4, nb);
}

// Phase 2 (after a cluster barrier): the unit's statistics (every CTA's, read through
// distributed shared memory), this CTA's window scores and the pooled scores of the
// blocks it owns, as ranking keys in this CTA's keys[b] and as floats in sq_blk.
__device__ __forceinline__ void pool_blocks(const LayerState& s, int u, const Geometry& geo, int rank, int CS,
                                            const Smem& m, SelShared& sh) {
  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x;
  const int G = s.G, wpc = s.score_wpc, nc = geo.nc, nb = geo.nb;
  const int i0 = rank * wpc;
  float* zs = m.zs;
  float* sqs = m.sqs;
  uint32_t* keys = m.keys;
  // ---------------- 2. unit statistics, window scores, pooled block maxima
  if (tid < G) {  // all CTAs' statistics for head tid, requested at once
    float mr[kMaxScoreCluster], sr[kMaxScoreCluster];
#pragma unroll
    for (int r = 0; r < kMaxScoreCluster; ++r) {
      mr[r] = r < CS ? *cluster.map_shared_rank(&sh.Mloc[tid], r) : -INFINITY;
      sr[r] = r < CS ? *cluster.map_shared_rank(&sh.Sloc[tid], r) : 0.f;
    }
    float M = -INFINITY;
#pragma unroll
    for (int r = 0; r < kMaxScoreCluster; ++r) M = fmaxf(M, mr[r]);
    float S = 0.f;
#pragma unroll
    for (int r = 0; r < kMaxScoreCluster; ++r)
      if (mr[r] > -INFINITY) S += sr[r] * expf(mr[r] - M);
    sh.Mh[tid] = M;
    sh.invS[tid] = 1.f / S;
  }
  __syncthreads();
  const int i1 = min(i0 + wpc, nc);
  for (int wl = tid; wl < i1 - i0; wl += blockDim.x) {
    float acc = 0.f;
    for (int h = 0; h < G; ++h) acc += expf(zs[h * wpc + wl] - sh.Mh[h]) * sh.invS[h];
    sqs[wl] = acc;
  }
  if (tid == 0) {
    float acc = 0.f;
    for (int h = 0; h < G; ++h) acc += expf(sh.zx[h] - sh.Mh[h]) * sh.invS[h];
    sh.sqx = (i0 >= 1 && i0 - 1 < nc) ? acc : -INFINITY;
  }
  __syncthreads();
  int b0, b1;
  owned_blocks(s, nb, rank, CS, b0, b1);
  for (int b = b0 + tid; b < b1; b += blockDim.x) {
    const int wlo = max(4 * b - 1, 0), whi = min(4 * b + 3, nc - 1);
    float mx = -INFINITY;
    for (int i = wlo; i <= whi; ++i) mx = fmaxf(mx, i < i0 ? sh.sqx : sqs[i - i0]);
    keys[b] = orderable(mx);
    s.sq_blk[(size_t)u * s.nb_max + b] = mx;
  }
  __syncthreads();
}

// Phase 2b (right after phase 2): this CTA's k_q best candidate blocks to the leader, or
// with to_all to every CTA of the cluster (each then selects on its own).
__device__ __forceinline__ void rank_local(const LayerState& s, const Geometry& geo, int rank, int CS,
                                           const Smem& m, SelShared& sh, bool to_all = false) {
  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x;
  const int nb = geo.nb;
  float* zs = m.zs;
  uint32_t* keys = m.keys;
  uint32_t* cand_key = m.cand_key;
  int32_t* cand_blk = m.cand_blk;
  // ---------------- 2b. each CTA ranks the candidate blocks it owns (a contiguous range);
  // its k_q best go to the leader, which then ranks only those (at most 8 * k_q)
  const int ws = geo.ws, kq = s.k_q;
  {
    int ob0, ob1;
    owned_blocks(s, nb, rank, CS, ob0, ob1);
    const int cb0 = max(ob0, s.sink), cb1 = min(ob1, ws);
    const int nown = max(cb1 - cb0, 0);
    const int ndst = to_all ? CS : 1;
    if (nown > kSortRankMin && kq > 0 && kq <= 32) {
      // many owned candidates: every warp sorts chunks of 32 composite keys and keeps the best 32
      // (bitonic sort and merge in registers), then warp 0 merges the warps' lists; its first
      // k_q lanes hold the winners in order
      const int lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
      unsigned long long best = 0ull;  // below every real key (whose block field, all ones minus b, is never 0)
      for (int base = warp * 32; base < nown; base += nwarps * 32) {
        const int i = base + lane;
        const unsigned long long x = i < nown ? rank_key(keys[cb0 + i], cb0 + i) : 0ull;
        best = warp_merge_top(best, warp_sort_desc(x));
      }
      unsigned long long* wbest = reinterpret_cast<unsigned long long*>(zs);  // z is no longer needed
      wbest[warp * 32 + lane] = best;
      __syncthreads();
      if (warp == 0) {
        unsigned long long a = wbest[lane];
        for (int w = 1; w < nwarps; ++w) a = warp_merge_top(a, wbest[w * 32 + lane]);
        if (lane < min(kq, nown))
          for (int d = 0; d < ndst; ++d) {
            cluster.map_shared_rank(cand_key, d)[rank * kq + lane] = (uint32_t)(a >> 32);
            cluster.map_shared_rank(cand_blk, d)[rank * kq + lane] = (int32_t)(0xFFFFFFFFu - (uint32_t)a);
          }
      }
    } else {
      unsigned long long* lk = reinterpret_cast<unsigned long long*>(zs);  // z is no longer needed
      for (int i = tid; i < nown; i += blockDim.x) lk[i] = rank_key(keys[cb0 + i], cb0 + i);
      __syncthreads();
      for (int i = tid; i < nown && kq > 0; i += blockDim.x) {
        const unsigned long long ki = lk[i];
        const int r = count_larger(lk, nown, ki);
        if (r < kq)
          for (int d = 0; d < ndst; ++d) {
            cluster.map_shared_rank(cand_key, d)[rank * kq + r] = (uint32_t)(ki >> 32);
            cluster.map_shared_rank(cand_blk, d)[rank * kq + r] = cb0 + i;
          }
      }
    }
    if (tid < ndst) *cluster.map_shared_rank(&sh.cand_n[rank], tid) = min(nown, max(kq, 0));
  }
}

// Phase 3a, in a CTA holding every CTA's local winners (after a cluster barrier and
// cp_async_wait_all): candidate flags and the query-aware picks Q (flags F_Q).
__device__ __forceinline__ void leader_query(const LayerState& s, int u, const Geometry& geo, int CS,
                                             const Smem& m, SelShared& sh) {
  const int tid = threadIdx.x;
  const int nb = geo.nb, ws = geo.ws, kq = s.k_q;
  float* zs = m.zs;
  uint32_t* cand_key = m.cand_key;
  int32_t* cand_blk = m.cand_blk;
  uint8_t* flags = m.flags;
  // ---------------- 3. selection by the leader
  for (int b = tid; b < nb; b += blockDim.x) flags[b] = (b >= s.sink && b < ws) ? F_CAND : 0;
  __syncthreads();
  // query-aware: gather the CTAs' winners into one list of composite keys and rank them
  unsigned long long* ck = reinterpret_cast<unsigned long long*>(zs);
  int* cofs = sh.cofs;
  if (tid == 0) {
    int o = 0;
    for (int r = 0; r < CS; ++r) {
      cofs[r] = o;
      o += sh.cand_n[r];
    }
    cofs[CS] = o;
  }
  __syncthreads();
  const int ncand = cofs[CS];
  for (int idx = tid; idx < CS * kq; idx += blockDim.x) {
    const int ri = idx / kq, j = idx % kq;
    if (j < sh.cand_n[ri]) ck[cofs[ri] + j] = rank_key(cand_key[idx], cand_blk[idx]);
  }
  __syncthreads();
  for (int i = tid; i < ncand; i += blockDim.x) {
    const unsigned long long ki = ck[i];
    if (count_larger(ck, ncand, ki) < kq) flags[0xFFFFFFFFu - (uint32_t)ki] |= F_Q;
  }
  __syncthreads();
}

// Phase 3b: the query-agnostic picks E, the selection S and the slots of its new blocks.
// The writer (one CTA per unit) also stores the eviction update, slot tables, fetch list,
// selection lists and statistics; every CTA that runs it on the same inputs reaches the
// same selection.  deal(pos, b, slot, isnew, dp, kind) is called for each selected block b at
// list position pos < cap, with its slot (as published), its dealing position dp (the blocks
// without a slot first, then the rest, each in block order) and its kind (0 sink, 1 window,
// 2 query-aware, 3 query-agnostic).  Returns |S|.
template <typename Deal>
__device__ __forceinline__ int leader_rest(const LayerState& s, int u, const Geometry& geo, const Smem& m,
                                           SelShared& sh, int my_slot_blk, bool writer, Deal deal) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nb = geo.nb, ws = geo.ws;
  float* zs = m.zs;
  uint32_t* keys = m.keys;
  float* sek = m.sek;
  int32_t* b2s = m.b2s;
  uint32_t* evw = m.evw;
  uint8_t* flags = m.flags;
  // query-agnostic: candidates outside Q never dropped before, ranked by pooled s^e
  const int per = (nb + blockDim.x - 1) / blockDim.x;
  const int lo = min(tid * per, nb), hi = min(lo + per, nb);
  int nel = 0;
  for (int b = lo; b < hi; ++b) {
    const bool evb = (evw[b >> 5] >> (b & 31)) & 1u;
    if ((flags[b] & F_CAND) && !(flags[b] & F_Q) && !evb) {
      flags[b] |= F_ELIG;
      ++nel;
    }
  }
  // the previous selection's context length: the latest one any cache slot served (-1: none)
  const int my_lu = tid < s.cslots ? m.lu[tid] : -1;
  {
    const int v = warp_max(my_lu);
    if (lane == 0) sh.lumax[warp] = v;
  }
  int n_elig;
  int epos = block_scan_excl(nel, sh.scan, &n_elig);  // its barriers also publish lumax
  int T_prev = -1;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) T_prev = max(T_prev, sh.lumax[w]);
  // a block of the previous selection holds a slot that served it then
  auto in_prev = [&](int b) {
    const int sl = b2s[b];
    return T_prev >= 0 && sl >= 0 && sl < s.cslots && m.lu[sl] == T_prev;
  };
  if (n_elig <= s.k_e) {
    for (int b = lo; b < hi; ++b)
      if (flags[b] & F_ELIG) flags[b] |= F_E;
  } else if (n_elig <= 1024 && !s.test_radix) {
    unsigned long long* ek = reinterpret_cast<unsigned long long*>(zs);
    for (int b = lo; b < hi; ++b)
      if (flags[b] & F_ELIG) ek[epos++] = rank_key(orderable(sek[b]), b);
    __syncthreads();
    for (int i = tid; i < n_elig; i += blockDim.x) {
      const unsigned long long ki = ek[i];
      if (count_larger(ek, n_elig, ki) < s.k_e) flags[0xFFFFFFFFu - (uint32_t)ki] |= F_E;
    }
  } else {  // many eligible blocks (a first selection over a long context): radix select
    for (int b = tid; b < nb; b += blockDim.x) keys[b] = orderable(sek[b]);
    __syncthreads();
    if (warp == 0) warp_topk(keys, flags, nb, s.k_e, F_ELIG, F_E, sh.hist);
  }
  __syncthreads();

  // selection S and the blocks without a slot; contiguous per-thread ranges keep block order
  int nD = 0, nE = 0, nDnew = 0, nS = 0, nNew = 0;
  for (int b = lo; b < hi; ++b) {
    uint8_t f = flags[b];
    const bool inS = b < geo.ns || b >= ws || (f & (F_Q | F_E));
    if (inS) {
      f |= F_S;
      ++nS;
      if (b2s[b] < 0) {
        f |= F_NEW;
        ++nNew;
      }
    }
    if (f & (F_Q | F_E)) {
      ++nD;
      if (!in_prev(b)) ++nDnew;
    }
    if (f & F_E) ++nE;
    flags[b] = f;
  }
  __syncthreads();
  // sticky eviction: candidates outside D are dropped for good (a warp ballot per 32 blocks)
  for (int w = warp; w < (nb + 31) / 32; w += (int)(blockDim.x >> 5)) {
    const int b = 32 * w + lane;
    const uint32_t bits =
        __ballot_sync(0xffffffffu, b < nb && (flags[b] & F_CAND) && !(flags[b] & (F_Q | F_E)));
    if (writer && lane == 0 && (bits & ~evw[w])) s.evicted[(size_t)u * s.ev_words + w] = evw[w] | bits;
  }
  // one scan of three counts (each at most 256, 10 bits apiece): cache slots open to new blocks
  // (empty, or holding a block outside the selection), blocks without a slot, selected blocks
  int32_t* sblk = s.slot_blk + (size_t)u * s.cslots;
  const bool own = tid < s.cslots;
  const bool holds_sel = own && my_slot_blk >= 0 && my_slot_blk < nb && (flags[my_slot_blk] & F_S);
  const int is_open = (own && !holds_sel) ? 1 : 0;
  int packed_total;
  const int packed = block_scan_excl(is_open | (nNew << 10) | (nS << 20), sh.scan, &packed_total);
  const int n_open = packed_total & 1023;
  const int new_before = (packed >> 10) & 1023, n_new_all = (packed_total >> 10) & 1023;
  int new_rank = new_before, n_new = n_new_all;
  int pos = packed >> 20;
  const int total_S = packed_total >> 20;
  if (n_new > n_open) {  // cannot happen when the cache holds a whole selection; guard the tables anyway
    if (writer && tid == 0) atomicOr(s.err, kErrBounds);
    n_new = n_open;
  }
  // the open slots the new blocks take: every one when there are as many, else the n_new least
  // recently selected (an empty slot counts as never selected; ties to the lower slot); the
  // others keep their blocks for later steps.  They are taken in ascending slot order.
  bool take = is_open && n_new > 0;
  int take_rank = packed & 1023;  // this slot's rank among the open ones
  if (n_new > 0 && n_new < n_open) {
    const uint32_t key = ((uint32_t)(my_lu + 1) << 9) | (uint32_t)tid;
    if (own) sh.okey[tid] = is_open ? key : 0xFFFFFFFFu;
    __syncthreads();
    if (is_open) {
      int r = 0;
#pragma unroll 8
      for (int j = 0; j < s.cslots; ++j) r += sh.okey[j] < key ? 1 : 0;
      take = r < n_new;
    }
    int n_take;
    take_rank = block_scan_excl(take ? 1 : 0, sh.scan, &n_take);
  }
  if (take) sh.free_by_rank[take_rank] = tid;
  int32_t* b2s_g = s.blk2slot + (size_t)u * s.nb_max;
  if (writer && take && my_slot_blk >= 0) {  // the block replaced in this slot is no longer cached
    if (my_slot_blk < s.nb_max) b2s_g[my_slot_blk] = -1;
    else atomicOr(s.err, kErrBounds);
  }
  __syncthreads();  // free_by_rank complete
  int32_t* fl = s.fetch + (size_t)u * s.cap * 2;
  for (int b = lo; b < hi; ++b) {
    if (!(flags[b] & F_NEW)) continue;
    if (new_rank < n_new) {
      const int slot = sh.free_by_rank[new_rank];
      b2s[b] = slot;
      if (writer) {
        b2s_g[b] = slot;
        sblk[slot] = b;
        fl[2 * new_rank] = b;
        fl[2 * new_rank + 1] = slot;
      }
    }
    ++new_rank;
  }
  // every slot that now holds a selected block served this selection
  if (writer && (holds_sel || take)) s.last_used[(size_t)u * s.cslots + tid] = geo.T;
  // ascending selection list with kinds, slots and the fetched marks (a thread's own blocks:
  // their slots were assigned just above by the same thread)
  int32_t* sel = s.sel + (size_t)u * s.cap;
  int32_t* kind = s.sel_kind + (size_t)u * s.cap;
  int32_t* sslot = s.sel_slot + (size_t)u * s.cap;
  int32_t* snew = s.sel_new + (size_t)u * s.cap;
  int nw_before = new_before;  // blocks without a slot ahead of b in block order
  for (int b = lo; b < hi; ++b) {
    const uint8_t f = flags[b];
    if (!(f & F_S)) continue;
    const bool isnew = f & F_NEW;
    if (pos < s.cap) {
      const int slot = (s.test_bad_slot && u == 0 && pos == 0) ? s.cslots : b2s[b];  // test hook
      const int kd = (f & F_Q) ? 2 : (f & F_E) ? 3 : (b < geo.ns ? 0 : 1);
      if (writer) {
        sel[pos] = b;
        kind[pos] = kd;
        sslot[pos] = slot;
        snew[pos] = isnew ? 1 : 0;
      }
      deal(pos, b, slot, isnew, isnew ? nw_before : n_new_all + pos - nw_before, kd);
    } else if (writer) {
      atomicOr(s.err, kErrBounds);
    }
    if (isnew) ++nw_before;
    ++pos;
  }
  if (!writer) return total_S;
  for (int i = total_S + tid; i < s.cap; i += blockDim.x) {
    sel[i] = -1;
    kind[i] = -1;
    sslot[i] = -1;
    snew[i] = 0;
  }
  // unit totals: |D|, |D \ S_prev|, |E|, whether there was a previous selection
  int4 v = make_int4(nD, nDnew, nE, T_prev >= 0 ? 1 : 0);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
    v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
    v.z += __shfl_xor_sync(0xffffffffu, v.z, o);
    v.w += __shfl_xor_sync(0xffffffffu, v.w, o);
  }
  if (lane == 0) sh.wsum[warp] = v;
  __syncthreads();
  if (tid == 0) {
    int4 t = sh.wsum[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
      t.x += sh.wsum[w].x;
      t.y += sh.wsum[w].y;
      t.z += sh.wsum[w].z;
      t.w += sh.wsum[w].w;
    }
    const int sumD = t.x, sumDnew = t.y, sumE = t.z, had_prev = t.w > 0;
    s.n_sel[u] = min(total_S, s.cap);
    s.n_fetch[u] = n_new;
    s.gamma[2 * u] = sumD - sumDnew;
    s.gamma[2 * u + 1] = sumD;
    atomicAdd(&s.stats->selections, 1ull);
    atomicAdd(&s.stats->blocks_fetched, (unsigned long long)n_new);
    if (sumE < s.k_e) atomicAdd(&s.stats->short_selections, 1ull);
    if (had_prev && sumD > 0) {
      atomicAdd(&s.stats->gamma_samples, 1ull);
      atomicAdd(&s.stats->gamma_num, (unsigned long long)(sumD - sumDnew));
      atomicAdd(&s.stats->gamma_den, (unsigned long long)sumD);
      const float gmm = (float)(sumD - sumDnew) / (float)sumD;
      atomicMin(&s.stats->gamma_min_bits, __float_as_uint(gmm));
    }
  }
  return total_S;
}

// Phase 3 (after a cluster barrier and cp_async_wait_all), in a CTA that holds every CTA's
// local winners: the selection; the writer also stores its global state (leader_rest).
template <typename Deal>
__device__ __forceinline__ int leader_select(const LayerState& s, int u, const Geometry& geo, int CS,
                                             const Smem& m, SelShared& sh, int my_slot_blk, bool writer,
                                             Deal deal) {
  leader_query(s, u, geo, CS, m, sh);
  return leader_rest(s, u, geo, m, sh, my_slot_blk, writer, deal);
}

}  // namespace selcore

}  // namespace nosa
