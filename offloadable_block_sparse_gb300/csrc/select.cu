// a2-a4: fused scorer, two-part selector, set difference and fetch list.
//
// One thread-block cluster per unit: CTA r of the cluster scores compressed
// windows [r*wpc, (r+1)*wpc).
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
// requested at kernel start and arrive while step 1 runs.
#include <cooperative_groups.h>

#include "nosa_internal.cuh"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace nosa {

namespace {

constexpr uint8_t F_CAND = 1, F_ELIG = 2, F_Q = 4, F_E = 8, F_S = 16, F_NEW = 32;
constexpr uint32_t kKeyNegInf = 0x007FFFFFu;  // orderable(-inf)
constexpr int kMaxScoreCluster = 8;

struct SelShared {
  int cand_n[kMaxScoreCluster];  // leader: local winners per cluster CTA
  int scan[32];
  int hist[256];
  int free_by_rank[256];
  float cmax[kScoreWarps][kMaxGroup];
  float Mloc[kMaxGroup], Sloc[kMaxGroup];  // this CTA's softmax statistics (read remotely)
  float Mh[kMaxGroup], invS[kMaxGroup];    // the unit's statistics
  int4 wsum[kScoreWarps];
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

// Floats of the first shared-memory region: the window logits, later reused for
// 64-bit ranking keys (up to 8 * k_q gathered winners, or one per block).
__host__ __device__ inline int zs_floats(const LayerState& s) {
  const int keys64 = 2 * (kMaxScoreCluster * s.k_q > s.nb_max ? kMaxScoreCluster * s.k_q : s.nb_max);
  return kMaxGroup * s.score_wpc > keys64 ? kMaxGroup * s.score_wpc : keys64;
}

__device__ __forceinline__ float from_orderable(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Top-k over the blocks whose flag has `valid` set, run by one warp: sets `mark`
// on the k largest keys, ties to the lower block index.  Radix select on the
// keys' offsets from the smallest valid key, 8-bit digits taken from the
// highest bit of (max - min) down, so the digits spread over the actual range
// of the scores (pooled scores share their high bits) and the shared-memory
// histogram atomics rarely collide; the bins are scanned with warp shuffles.  The keys
// equal to the k-th largest are then taken in ascending block order by ballot.
__device__ void warp_topk(const uint32_t* keys, uint8_t* flags, int n, int k, uint8_t valid, uint8_t mark,
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

}  // namespace

// grid (cluster size, U) with clusters (cluster size, 1, 1); 256 threads.
// Dynamic shared memory: z[kMaxGroup][wpc] and sq[wpc] floats (every CTA), then
// for the leader keys[nb_max], se[nb_max], b2s[nb_max], eviction words, flags[nb_max].
__global__ void __launch_bounds__(kScoreThreads) score_select_kernel(LayerState s, const uint16_t* __restrict__ q) {
  extern __shared__ __align__(16) unsigned char dsm[];
  __shared__ SelShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank(), CS = (int)cluster.num_blocks();
  const int u = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gr = lane >> 2, t4 = lane & 3;
  const int G = s.G, wpc = s.score_wpc;
  float* zs = reinterpret_cast<float*>(dsm);                      // [kMaxGroup][wpc], later ranking keys
  float* sqs = zs + zs_floats(s);                                 // [wpc]
  uint32_t* keys = reinterpret_cast<uint32_t*>(sqs + wpc);        // leader: [nb_max]
  float* sek = reinterpret_cast<float*>(keys + s.nb_max);         // leader: [nb_max] pooled s^e
  int32_t* b2s = reinterpret_cast<int32_t*>(sek + s.nb_max);      // leader: [nb_max] block -> slot
  uint32_t* evw = reinterpret_cast<uint32_t*>(b2s + s.nb_max);    // leader: [ev_words]
  uint32_t* cand_key = evw + s.ev_words;                          // leader: [8][k_q] local winners' keys
  int32_t* cand_blk = reinterpret_cast<int32_t*>(cand_key + kMaxScoreCluster * s.k_q);  // [8][k_q]
  int32_t* eblk = cand_blk + kMaxScoreCluster * s.k_q;             // leader: [nb_max] eligible blocks
  uint8_t* flags = reinterpret_cast<uint8_t*>(eblk + s.nb_max);   // leader: [nb_max]

  // q fragments first: they do not depend on the context length.  The k order in
  // each 32-dim chunk is permuted identically for A (K~ rows) and B (q), so a
  // thread loads 16 contiguous bytes per row and a warp load covers whole sectors.
  uint4 qf[4];
  {
    const uint16_t* qh = q + ((size_t)u * G + min(gr, G - 1)) * kHeadDim;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      qf[c] = gr < G ? *reinterpret_cast<const uint4*>(qh + 32 * c + 8 * t4) : make_uint4(0, 0, 0, 0);
  }
  pdl_wait();               // the append kernel's context length, keys and scores are needed from here
  pdl_launch_dependents();  // the attention kernel may start its own prologue
  const Geometry geo = geometry(*s.T, s.nw, s.sink);
  const int nc = geo.nc, nb = geo.nb;
  const int i0 = rank * wpc;  // first window of this CTA

  // leader: request the selection's inputs now as asynchronous copies into shared
  // memory; they land while the scoring runs (waited for before the selection)
  int my_slot_blk = -1;
  if (rank == 0) {
    const float* seg = s.se_blk + (size_t)u * s.nb_max;
    const int32_t* b2g = s.blk2slot + (size_t)u * s.nb_max;
    const uint32_t* evg = s.evicted + (size_t)u * s.ev_words;
    for (int b = tid; b < nb; b += blockDim.x) {
      keys[b] = kKeyNegInf;
      cp_async_4(smem_u32(sek + b), seg + b);
      cp_async_4(smem_u32(b2s + b), b2g + b);
    }
    for (int w = tid; w < (nb + 31) / 32; w += blockDim.x) cp_async_4(smem_u32(evw + w), evg + w);
    cp_async_commit();
    if (tid < s.cap) my_slot_blk = s.slot_blk[(size_t)u * s.cap + tid];
  }

  // ---------------- 1. z for this CTA's windows, per-head max
  const float scale = s.scale;
  float mx[2] = {-INFINITY, -INFINITY};
  const int tiles = wpc / (16 * kScoreWarps);
  for (int t0 = 0; t0 < tiles; t0 += 2) {
    uint4 a[2][2][4];
#pragma unroll
    for (int tl = 0; tl < 2; ++tl)
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
    for (int tl = 0; tl < 2; ++tl) {
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
    for (int w = 0; w < kScoreWarps; ++w) m = fmaxf(m, sh.cmax[w][tid]);
    sh.Mloc[tid] = m;
  }
  __syncthreads();
  // sum of exp per head over this CTA's windows: warp w handles head w
  if (warp < G) {
    const float M = sh.Mloc[warp];
    float e = 0.f;
    if (M > -INFINITY)
      for (int wl = lane; wl < wpc; wl += 32) e += expf(zs[warp * wpc + wl] - M);  // exp(-inf) = 0
    e = warp_sum(e);
    if (lane == 0) sh.Sloc[warp] = e;
  }
  cluster.sync();  // every CTA's statistics (and the leader's key init) are visible

  // ---------------- 2. unit statistics, window scores, pooled block maxima -> leader
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
  __syncthreads();
  if (i1 > i0) {
    uint32_t* lkeys = cluster.map_shared_rank(keys, 0);
    const int b_lo = (kCmpStride * i0) / kBlock, b_hi = (kCmpStride * (i1 - 1) + kCmpKernel - 1) / kBlock;
    for (int b = b_lo + tid; b <= b_hi; b += blockDim.x) {
      const int wlo = max(4 * b - 1, i0), whi = min(4 * b + 3, i1 - 1);
      float m = -INFINITY;
      for (int i = wlo; i <= whi; ++i) m = fmaxf(m, sqs[i - i0]);
      if (wlo <= whi) atomicMax(lkeys + b, orderable(m));
    }
  }
  cluster.sync();  // block maxima have landed in the leader; remote reads are done

  // ---------------- 2b. each CTA ranks the candidate blocks it owns (a contiguous range);
  // its k_q best go to the leader, which then ranks only those (at most 8 * k_q)
  const int ws = geo.ws, kq = s.k_q;
  {
    const int nbpc = (nb + CS - 1) / CS;
    const int ob0 = min(rank * nbpc, nb), ob1 = min(ob0 + nbpc, nb);
    const int cb0 = max(ob0, s.sink), cb1 = min(ob1, ws);
    const int nown = max(cb1 - cb0, 0);
    unsigned long long* lk = reinterpret_cast<unsigned long long*>(zs);  // z is no longer needed
    const uint32_t* lkeys = cluster.map_shared_rank(keys, 0);
    for (int i = tid; i < nown; i += blockDim.x) lk[i] = rank_key(lkeys[cb0 + i], cb0 + i);
    __syncthreads();
    uint32_t* ckey = cluster.map_shared_rank(cand_key, 0);
    int32_t* cblk = cluster.map_shared_rank(cand_blk, 0);
    for (int i = tid; i < nown && kq > 0; i += blockDim.x) {
      const unsigned long long ki = lk[i];
      const int r = count_larger(lk, nown, ki);
      if (r < kq) {
        ckey[rank * kq + r] = (uint32_t)(ki >> 32);
        cblk[rank * kq + r] = cb0 + i;
      }
    }
    if (tid == 0) *cluster.map_shared_rank(&sh.cand_n[rank], 0) = min(nown, max(kq, 0));
  }
  cluster.sync();  // the local winners have landed in the leader
  if (rank != 0) return;
  cp_async_wait_all();  // the leader's early copies (pooled s^e, slot map, eviction words)

  // ---------------- 3. selection by the leader
  for (int b = tid; b < nb; b += blockDim.x) {
    s.sq_blk[(size_t)u * s.nb_max + b] = from_orderable(keys[b]);
    flags[b] = (b >= s.sink && b < ws) ? F_CAND : 0;
  }
  __syncthreads();
  // query-aware: gather the CTAs' winners into one list of composite keys and rank them
  unsigned long long* ck = reinterpret_cast<unsigned long long*>(zs);
  __shared__ int cofs[kMaxScoreCluster + 1];
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
  int n_elig;
  int epos = block_scan_excl(nel, sh.scan, &n_elig);
  if (n_elig <= s.k_e) {
    for (int b = lo; b < hi; ++b)
      if (flags[b] & F_ELIG) flags[b] |= F_E;
  } else if (n_elig <= 1024) {
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
      if (f & F_NEW) ++nDnew;
    }
    if (f & F_E) ++nE;
    flags[b] = f;
  }
  __syncthreads();
  // sticky eviction: candidates outside D are dropped for good
  for (int w = tid; w < (nb + 31) / 32; w += blockDim.x) {
    uint32_t bits = 0;
    for (int j = 0; j < 32; ++j) {
      const int b = 32 * w + j;
      if (b < nb && (flags[b] & F_CAND) && !(flags[b] & (F_Q | F_E))) bits |= 1u << j;
    }
    if (bits & ~evw[w]) s.evicted[(size_t)u * s.ev_words + w] = evw[w] | bits;
  }
  // free slots: empty, or holding a block that left the selection (ascending)
  int32_t* sblk = s.slot_blk + (size_t)u * s.cap;
  const int is_free = tid < s.cap && !(my_slot_blk >= 0 && my_slot_blk < nb && (flags[my_slot_blk] & F_S));
  int n_free;
  const int free_rank = block_scan_excl(is_free, sh.scan, &n_free);
  if (is_free) sh.free_by_rank[free_rank] = tid;
  int n_new;
  int new_rank = block_scan_excl(nNew, sh.scan, &n_new);
  if (n_new > n_free) {  // cannot happen when cap >= |S|; guard the slot table anyway
    if (tid == 0) atomicOr(s.err, kErrBounds);
    n_new = n_free;
  }
  int32_t* b2s_g = s.blk2slot + (size_t)u * s.nb_max;
  if (is_free && my_slot_blk >= 0) {
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
      b2s_g[b] = slot;
      sblk[slot] = b;
      fl[2 * new_rank] = b;
      fl[2 * new_rank + 1] = slot;
    }
    ++new_rank;
  }
  if (is_free && free_rank >= n_new) sblk[tid] = -1;
  __syncthreads();
  // ascending selection list with kinds, slots and the fetched marks
  int total_S;
  int pos = block_scan_excl(nS, sh.scan, &total_S);
  int32_t* sel = s.sel + (size_t)u * s.cap;
  int32_t* kind = s.sel_kind + (size_t)u * s.cap;
  int32_t* sslot = s.sel_slot + (size_t)u * s.cap;
  int32_t* snew = s.sel_new + (size_t)u * s.cap;
  for (int b = lo; b < hi; ++b) {
    const uint8_t f = flags[b];
    if (!(f & F_S)) continue;
    if (pos < s.cap) {
      sel[pos] = b;
      kind[pos] = (f & F_Q) ? 2 : (f & F_E) ? 3 : (b < geo.ns ? 0 : 1);
      sslot[pos] = (s.test_bad_slot && u == 0 && pos == 0) ? s.cap : b2s[b];  // test hook
      snew[pos] = (f & F_NEW) ? 1 : 0;
    } else {
      atomicOr(s.err, kErrBounds);
    }
    ++pos;
  }
  for (int i = total_S + tid; i < s.cap; i += blockDim.x) {
    sel[i] = -1;
    kind[i] = -1;
    sslot[i] = -1;
    snew[i] = 0;
  }
  // unit totals: |D|, |D \ S_prev|, |E|, whether any block was resident before
  int4 v = make_int4(nD, nDnew, nE, (tid < s.cap && my_slot_blk >= 0) ? 1 : 0);
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
    for (int w = 1; w < kScoreWarps; ++w) {
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
}

size_t score_select_smem(const LayerState& s) {
  return sizeof(float) * ((size_t)zs_floats(s) + s.score_wpc) + 4 * sizeof(uint32_t) * s.nb_max +
         sizeof(uint32_t) * s.ev_words + 2 * sizeof(uint32_t) * kMaxScoreCluster * s.k_q + s.nb_max + 16;
}

cudaError_t init_score_select(const LayerState& s) {
  return cudaFuncSetAttribute(score_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)score_select_smem(s));
}

cudaError_t launch_score_select(const LayerState& s, const uint16_t* q, bool pdl, cudaStream_t st) {
  return launch_ex(score_select_kernel, dim3(s.score_chunks, s.U), dim3(kScoreThreads), score_select_smem(s), st,
                   pdl, s.score_chunks, s, q);
}

}  // namespace nosa
