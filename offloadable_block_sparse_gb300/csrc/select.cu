// a2-a4: fused scorer, two-part selector, set difference and fetch list.
//
// Phase 1 (every CTA): z_{h,i} = q_h . K~_i * scale for a chunk of compressed
// windows, on the tensor cores (mma.sync m16n8k16, windows as M, the GQA
// group's heads as N), plus the chunk's per-head softmax statistics.
// Phase 2 (last CTA of each unit, by atomic ticket): per-head softmax over all
// windows summed over the group (SparDA summary, "lightweight design": the
// block selector aggregates the group's heads through a softmax), max-pooled
// onto the 64-token blocks (NOSA explainer eq. 5-6); top-k_q query-aware
// blocks, then k_e blocks by the pooled eviction score among candidates never
// dropped before (wiki "How NOSA works": query-aware picks set to +inf, the
// rest filled by the query-agnostic score, never-reselect constraint); sink
// and window blocks; sticky eviction update; set difference against the
// block cache with ascending free-slot assignment (wiki "NOSI": set-difference
// kernel, only changed blocks are swapped).
#include "nosa_internal.cuh"
#include "ptx.cuh"

namespace nosa {

namespace {

constexpr uint8_t F_CAND = 1, F_ELIG = 2, F_Q = 4, F_E = 8, F_S = 16, F_NEW = 32;

struct SelShared {
  int scan[32];
  int hist[256];
  int free_by_rank[256];
  int digit, above, total, last;
  float cmax[kScoreWarps][kMaxGroup];
  float Mh[kMaxGroup], invS[kMaxGroup];
};

// Top-k over the blocks whose flag has `valid` set, run by one warp: sets `mark`
// on the k largest keys, ties to the lower block index.  Radix select on the
// 32-bit keys (4 passes of 8 bits; histogram in shared memory, bins scanned
// with warp shuffles), then the keys equal to the k-th largest are taken in
// ascending block order with ballots.  No block-wide barrier.
__device__ void warp_topk(const uint32_t* keys, uint8_t* flags, int n, int k, uint8_t valid, uint8_t mark,
                          int* hist) {
  const int lane = threadIdx.x & 31;
  if (k <= 0) return;
  int cnt = 0;
  for (int b = lane; b < n; b += 32) cnt += (flags[b] & valid) ? 1 : 0;
  cnt = warp_sum(cnt);
  if (cnt <= k) {
    for (int b = lane; b < n; b += 32)
      if (flags[b] & valid) flags[b] |= mark;
    __syncwarp();
    return;
  }
  uint32_t prefix = 0, pmask = 0;
  int need = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = lane; i < 256; i += 32) hist[i] = 0;
    __syncwarp();
    for (int b = lane; b < n; b += 32)
      if ((flags[b] & valid) && (keys[b] & pmask) == prefix) atomicAdd(&hist[(keys[b] >> shift) & 255], 1);
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
    pmask |= 255u << shift;
    __syncwarp();
  }
  // prefix is the k-th largest key; `need` keys equal to it are taken, lowest blocks first
  int taken = 0;
  for (int base = 0; base < n; base += 32) {
    const int b = base + lane;
    const bool v = b < n && (flags[b] & valid);
    const uint32_t key = v ? keys[b] : 0u;
    const bool tie = v && key == prefix;
    const unsigned int tm = __ballot_sync(0xffffffffu, tie);
    const int rank = taken + __popc(tm & ((1u << lane) - 1u));
    if ((v && key > prefix) || (tie && rank < need)) flags[b] |= mark;
    taken += __popc(tm);
  }
  __syncwarp();
}

}  // namespace

// grid (score_chunks, U), 256 threads.  Dynamic shared memory (phase 2): window
// scores, pooled s^e, block->slot map, radix keys, chunk stats, eviction words, flags.
__global__ void __launch_bounds__(kScoreThreads) score_select_kernel(LayerState s, const uint16_t* __restrict__ q) {
  extern __shared__ __align__(16) unsigned char dsm[];
  __shared__ SelShared sh;
  const int chunk = blockIdx.x, u = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gr = lane >> 2, t4 = lane & 3;
  const Geometry geo = geometry(*s.T, s.nw, s.sink);
  const int G = s.G, nc = geo.nc;

  // ---------------- phase 1: z for this chunk of windows
  // k order inside each 32-dim chunk is permuted identically for A (K~ rows) and
  // B (q), so each thread loads 16 contiguous bytes per row: lanes t4 of a row
  // cover 64 contiguous bytes and a warp load touches whole 32-byte sectors.
  uint4 qf[4];
  {
    const uint16_t* qh = q + ((size_t)u * G + gr) * kHeadDim;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      qf[c] = gr < G ? *reinterpret_cast<const uint4*>(qh + 32 * c + 8 * t4) : make_uint4(0, 0, 0, 0);
  }
  const float scale = s.scale;
  float z[kScoreTiles][4];
  int rowi[kScoreTiles][2];
  {
    uint4 a[kScoreTiles][2][4];
#pragma unroll
    for (int tl = 0; tl < kScoreTiles; ++tl) {
      const int base = chunk * kWindowsPerCta + (warp * kScoreTiles + tl) * 16;
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int r = base + gr + 8 * hr;
        rowi[tl][hr] = r;
        const uint16_t* kr = s.kt + ((size_t)u * s.nc_max + min(r, s.nc_max - 1)) * kHeadDim;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          a[tl][hr][c] = r < nc ? *reinterpret_cast<const uint4*>(kr + 32 * c + 8 * t4) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int tl = 0; tl < kScoreTiles; ++tl) {
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
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = rowi[tl][j >> 1];
        z[tl][j] = r < nc ? acc[j] * scale : -INFINITY;
      }
    }
  }
  // store z and the chunk's per-head max
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int tl = 0; tl < kScoreTiles; ++tl)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int h = 2 * t4 + (j & 1), r = rowi[tl][j >> 1];
      if (h < G && r < nc) s.zbuf[((size_t)u * G + h) * s.nc_max + r] = z[tl][j];
      mx[j & 1] = fmaxf(mx[j & 1], z[tl][j]);
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
    sh.Mh[tid] = m;
  }
  __syncthreads();
  float se[2] = {0.f, 0.f};
#pragma unroll
  for (int tl = 0; tl < kScoreTiles; ++tl)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float M = sh.Mh[2 * t4 + (j & 1)];
      if (z[tl][j] > -INFINITY) se[j & 1] += expf(z[tl][j] - M);
    }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    se[j] += __shfl_xor_sync(0xffffffffu, se[j], 4);
    se[j] += __shfl_xor_sync(0xffffffffu, se[j], 8);
    se[j] += __shfl_xor_sync(0xffffffffu, se[j], 16);
  }
  __syncthreads();
  if (gr == 0) {
    sh.cmax[warp][2 * t4] = se[0];
    sh.cmax[warp][2 * t4 + 1] = se[1];
  }
  __syncthreads();
  if (tid < G) {
    float ssum = 0.f;
    for (int w = 0; w < kScoreWarps; ++w) ssum += sh.cmax[w][tid];
    float* sp = s.spart + (((size_t)u * s.score_chunks + chunk) * kMaxGroup + tid) * 2;
    sp[0] = sh.Mh[tid];
    sp[1] = ssum;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned int t = atomicAdd(&s.tickets[u], 1u);
    sh.last = (t == (unsigned int)s.score_chunks - 1);
  }
  __syncthreads();
  if (!sh.last) return;
  __threadfence();
  if (tid == 0) s.tickets[u] = 0;

  // ---------------- phase 2: selection for unit u
  // Every global value the selection needs is requested up front (one memory
  // round trip); the rest runs from shared memory.
  const int nb = geo.nb, ws = geo.ws;
  const int nch = s.score_chunks;
  float* sqw = reinterpret_cast<float*>(dsm);                   // [nc_max] window scores
  float* sek = sqw + s.nc_max;                                  // [nb_max] pooled s^e
  int32_t* b2s = reinterpret_cast<int32_t*>(sek + s.nb_max);    // [nb_max] block -> slot
  uint32_t* keys = reinterpret_cast<uint32_t*>(b2s + s.nb_max); // [nb_max]
  float* sp = reinterpret_cast<float*>(keys + s.nb_max);        // [nch][G][2] chunk stats
  uint32_t* evw = reinterpret_cast<uint32_t*>(sp + nch * kMaxGroup * 2);  // [ev_words]
  uint8_t* flags = reinterpret_cast<uint8_t*>(evw + s.ev_words);          // [nb_max]
  const int per = (nb + blockDim.x - 1) / blockDim.x;
  const int lo = min(tid * per, nb), hi = min(lo + per, nb);
  const int words = (nb + 31) / 32;
  for (int idx = tid; idx < nch * G; idx += blockDim.x) {
    const int j = idx / G, h = idx % G;
    const float* p = s.spart + (((size_t)u * nch + j) * kMaxGroup + h) * 2;
    sp[(j * kMaxGroup + h) * 2] = __ldcg(p);
    sp[(j * kMaxGroup + h) * 2 + 1] = __ldcg(p + 1);
  }
  for (int b = lo; b < hi; ++b) {
    sek[b] = s.se_blk[(size_t)u * s.nb_max + b];
    b2s[b] = s.blk2slot[(size_t)u * s.nb_max + b];
  }
  for (int w = tid; w < words; w += blockDim.x) evw[w] = s.evicted[(size_t)u * s.ev_words + w];
  int32_t* sblk = s.slot_blk + (size_t)u * s.cap;
  const int my_slot_blk = tid < s.cap ? sblk[tid] : -1;
  __syncthreads();
  if (tid < G) {
    float M = -INFINITY;
    for (int j = 0; j < nch; ++j) M = fmaxf(M, sp[(j * kMaxGroup + tid) * 2]);
    float S = 0.f;
    for (int j = 0; j < nch; ++j) {
      const float mj = sp[(j * kMaxGroup + tid) * 2];
      if (mj > -INFINITY) S += sp[(j * kMaxGroup + tid) * 2 + 1] * expf(mj - M);
    }
    sh.Mh[tid] = M;
    sh.invS[tid] = 1.f / S;
  }
  __syncthreads();
  // s^q per window: the group's softmax probabilities summed over heads
  for (int i0 = tid; i0 < nc; i0 += 4 * blockDim.x) {
    float zv[4][kMaxGroup];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = i0 + r * blockDim.x;
#pragma unroll
      for (int h = 0; h < kMaxGroup; ++h)
        zv[r][h] = (h < G && i < nc) ? __ldcg(s.zbuf + ((size_t)u * G + h) * s.nc_max + i) : 0.f;
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = i0 + r * blockDim.x;
      if (i >= nc) continue;
      float acc = 0.f;
#pragma unroll
      for (int h = 0; h < kMaxGroup; ++h)
        if (h < G) acc += expf(zv[r][h] - sh.Mh[h]) * sh.invS[h];
      sqw[i] = acc;
    }
  }
  __syncthreads();
  // max-pool onto blocks; candidates lie strictly between the sink and the window
  for (int b = lo; b < hi; ++b) {
    const int wl = max(4 * b - 1, 0), wh = min(4 * b + 3, nc - 1);
    float m = -INFINITY;
    for (int i = wl; i <= wh; ++i) m = fmaxf(m, sqw[i]);
    s.sq_blk[(size_t)u * s.nb_max + b] = m;
    keys[b] = orderable(m);
    flags[b] = (b >= s.sink && b < ws) ? F_CAND : 0;
  }
  __syncthreads();
  if (warp == 0) warp_topk(keys, flags, nb, s.k_q, F_CAND, F_Q, sh.hist);
  __syncthreads();
  for (int b = lo; b < hi; ++b) {
    keys[b] = orderable(sek[b]);
    const bool evb = (evw[b >> 5] >> (b & 31)) & 1u;
    if ((flags[b] & F_CAND) && !(flags[b] & F_Q) && !evb) flags[b] |= F_ELIG;
  }
  __syncthreads();
  if (warp == 0) warp_topk(keys, flags, nb, s.k_e, F_ELIG, F_E, sh.hist);
  __syncthreads();

  // selection S, blocks without a slot
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
  for (int w = tid; w < words; w += blockDim.x) {
    uint32_t bits = 0;
    for (int j = 0; j < 32; ++j) {
      const int b = 32 * w + j;
      if (b < nb && (flags[b] & F_CAND) && !(flags[b] & (F_Q | F_E))) bits |= 1u << j;
    }
    if (bits & ~evw[w]) s.evicted[(size_t)u * s.ev_words + w] = evw[w] | bits;
  }
  // free slots: empty, or holding a block that left the selection (ascending)
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
  // ascending selection list with kinds and slots
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
      sslot[pos] = b2s[b];
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
  __shared__ int4 wsum[kScoreWarps];
  if (lane == 0) wsum[warp] = v;
  __syncthreads();
  if (tid == 0) {
    int4 t = wsum[0];
    for (int w = 1; w < kScoreWarps; ++w) {
      t.x += wsum[w].x;
      t.y += wsum[w].y;
      t.z += wsum[w].z;
      t.w += wsum[w].w;
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
  return sizeof(float) * s.nc_max + 3 * sizeof(uint32_t) * s.nb_max +
         sizeof(float) * s.score_chunks * kMaxGroup * 2 + sizeof(uint32_t) * s.ev_words + s.nb_max + 16;
}

cudaError_t init_score_select(const LayerState& s) {
  return cudaFuncSetAttribute(score_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)score_select_smem(s));
}

cudaError_t launch_score_select(const LayerState& s, const uint16_t* q, cudaStream_t st) {
  const size_t smem = score_select_smem(s);
  score_select_kernel<<<dim3(s.score_chunks, s.U), kScoreThreads, smem, st>>>(s, q);
  return cudaGetLastError();
}

}  // namespace nosa
