// NOSA_S sparse prefill: a prompt appended to an empty layer, every prompt position
// attended over its own block selection (NOSA wiki, "Results": NOSA_S is sparse in
// prefill as well as in decoding; NOSA wiki, "How NOSA works": the query-agnostic
// part never re-selects a block it dropped at an earlier step).  The selection for
// position t is the decode step's selection at T = t + 1 with the eviction state
// carried from position t - 1, so the positions are selected in order, and their
// attention then runs in one launch.
//
//   1. bulk append (append.cu): host store, eviction scores, compressed keys.
//   2a. prefill_query_kernel: the query-aware part of every position's selection at once
//      (it reads only the position's q and the windows complete at its T): scores over
//      those windows, the group softmax summed over heads, max-pooled onto the blocks, the
//      top-k_q candidates.  Each warp takes a few positions and walks the compressed keys.
//   2b. prefill_walk_kernel: one warp per unit makes the rest of every position's
//      selection in order: the k_e query-agnostic picks among the candidates never
//      dropped before (a short list ordered by pooled s^e) and the sticky eviction
//      update, with bitmaps over the blocks.  Each position's picks go to the caller's
//      scratch as two bitmaps (query-aware, query-agnostic).  The selection and eviction
//      state after the prompt are the ones the decode steps would have left; the cache
//      then holds exactly the last selection, its i-th block in slot i.
//   3. prefill_refresh_kernel: every cache slot gets its block's K/V from the prompt.
//   4. prefill_attend_tc_kernel: a CTA takes 128 / G consecutive positions of one unit (128
//      rows of position x q head), forms the union of their selections and streams those
//      blocks from the prompt's K and V (TMA, 128-byte swizzle); each block's scores and
//      its product with V run on the fifth-generation tensor cores (tcgen05, accumulators
//      in tensor memory), one thread per row does that row's masking and online softmax.
//      Positions share every block they have in common.
#include "attend_core.cuh"  // kStageBytes, the TMA and mbarrier helpers
#include "host.h"
#include "select_core.cuh"
#include "tc.cuh"

namespace nosa {

using namespace selcore;

constexpr int kPfMaxWords = 2048 / 32;  // block bitmap words per position (prompts of up to 131,072 tokens)
constexpr int kTcRowsQ = 128;           // rows of a query-aware tcgen05 tile: positions x q heads

// 2^x by the special-function unit (relative error about 2^-22; -inf gives 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------- 2a. query-aware picks, all positions
// The query-aware part of a position's selection depends only on its q and the windows complete
// at its T, not on the eviction state, so every position's k_q picks are made at once.
constexpr int kPqWarps = 8;

// grid (ceil(n / (8 PW)), U), 256 threads; dynamic shared memory [8 PW][nbn] pooled scores.
// Warp w takes positions tw .. tw + PW - 1 (tw = (8 blockIdx.x + w) PW), their q fragments in
// registers, and walks the unit's compressed keys in 16-window tiles twice (through L1, which the
// CTA's warps share): the first pass forms, per position and head, the maximum and the sum of
// exp of z_{h,i} = q_h . K~_i * scale (base 2) over the windows complete at the position's T
// (online); the second forms the group softmax summed over the heads per window and max-pools it onto the
// blocks each window overlaps.  Each position's k_q best candidate blocks (score, then lower
// block) go to qsel [U][n][nbw] as a bitmap over the blocks (nbw = ceil(nbn / 32) words).  The
// last position's pooled scores are also the layer's debug scores (sq_blk).
template <int PW>
__global__ void __launch_bounds__(kPqWarps * 32, 1)
    prefill_query_kernel(LayerState s, const uint16_t* __restrict__ q, uint32_t* __restrict__ qsel, int n, int nbn) {
  extern __shared__ uint32_t pool_sm[];
  __shared__ uint32_t qword_sm[kPqWarps][kPfMaxWords];
  const int u = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, t4 = lane & 3;
  const int G = s.G, kq = s.k_q;
  const int tw = (blockIdx.x * kPqWarps + warp) * PW;
  uint32_t* pooled = pool_sm + (size_t)warp * PW * nbn;
  pdl_wait();  // the bulk append wrote the compressed keys
  if (tw >= n) return;  // no CTA-wide barrier follows
  const int np = min(PW, n - tw);
  uint4 qf[PW][4];
  int nc[PW];
#pragma unroll
  for (int p = 0; p < PW; ++p) {
    const int t = min(tw + p, n - 1);
    nc[p] = geometry(t + 1, s.nw, s.sink).nc;
    // q of position t: head j of unit u is row (u * G + j) * n + t
    const uint16_t* qh = q + (((size_t)u * G + min(gr, G - 1)) * n + t) * kHeadDim;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      qf[p][c] = gr < G ? __ldg(reinterpret_cast<const uint4*>(qh + 32 * c + 8 * t4)) : make_uint4(0, 0, 0, 0);
  }
  for (int i = lane; i < PW * nbn; i += 32) pooled[i] = 0u;  // +0.0f: group scores are non-negative
  const int ncw = nc[np - 1];  // the warp's last position has the most windows
  const int ntiles = (ncw + 15) >> 4;
  const float scale2 = s.scale * 1.4426950408889634f;  // logits in base 2
  const uint16_t* kt = s.kt + (size_t)u * s.nc_max * kHeadDim;
  auto load_tile = [&](int tl, uint4 (&a)[2][4]) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = tl * 16 + gr + 8 * hr;
      const uint16_t* kr = kt + (size_t)(r < ncw ? r : 0) * kHeadDim;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        a[hr][c] = r < ncw ? __ldg(reinterpret_cast<const uint4*>(kr + 32 * c + 8 * t4)) : make_uint4(0, 0, 0, 0);
    }
  };
  // rows: windows tl*16 + gr (acc 0, 1) and + 8 (acc 2, 3); columns: heads 2 t4 (acc 0, 2), 2 t4 + 1
  auto logits = [&](const uint4 (&a)[2][4], const uint4 (&qq)[4], float (&acc)[4]) {
    acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t* r0 = reinterpret_cast<const uint32_t*>(&a[0][c]);
      const uint32_t* r1 = reinterpret_cast<const uint32_t*>(&a[1][c]);
      const uint32_t* qv = reinterpret_cast<const uint32_t*>(&qq[c]);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t af[4] = {r0[2 * hh], r1[2 * hh], r0[2 * hh + 1], r1[2 * hh + 1]};
        mma_16816(acc, af, qv[2 * hh], qv[2 * hh + 1]);
      }
    }
  };
  float M[PW][2], L[PW][2];
#pragma unroll
  for (int p = 0; p < PW; ++p) M[p][0] = M[p][1] = -INFINITY, L[p][0] = L[p][1] = 0.f;
  for (int tl = 0; tl < ntiles; ++tl) {  // pass 1: per (position, head) maximum and sum of exp
    uint4 a[2][4];
    load_tile(tl, a);
    const int w0 = tl * 16 + gr;
#pragma unroll
    for (int p = 0; p < PW; ++p) {
      if (p >= np) break;
      float acc[4];
      logits(a, qf[p], acc);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float z0 = w0 < nc[p] ? acc[j] * scale2 : -INFINITY;
        const float z1 = w0 + 8 < nc[p] ? acc[2 + j] * scale2 : -INFINITY;
        const float mn = fmaxf(M[p][j], fmaxf(z0, z1));
        if (mn > -INFINITY) {
          L[p][j] = (mn > M[p][j] ? L[p][j] * ex2(M[p][j] - mn) : L[p][j]) + ex2(z0 - mn) + ex2(z1 - mn);
          M[p][j] = mn;
        }
      }
    }
  }
  float inv[PW][2];
#pragma unroll
  for (int p = 0; p < PW; ++p)
#pragma unroll
    for (int j = 0; j < 2; ++j) {  // the lanes of one column hold different windows
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, M[p][j], o), lo = __shfl_xor_sync(0xffffffffu, L[p][j], o);
        const float mn = fmaxf(M[p][j], mo);
        if (mn > -INFINITY) {
          L[p][j] = (M[p][j] > -INFINITY ? L[p][j] * ex2(M[p][j] - mn) : 0.f) + (mo > -INFINITY ? lo * ex2(mo - mn) : 0.f);
          M[p][j] = mn;
        }
      }
      inv[p][j] = L[p][j] > 0.f ? 1.f / L[p][j] : 0.f;
    }
  for (int tl = 0; tl < ntiles; ++tl) {  // pass 2: group scores per window, max-pooled onto blocks
    uint4 a[2][4];
    load_tile(tl, a);
    const int w0 = tl * 16 + gr;
#pragma unroll
    for (int p = 0; p < PW; ++p) {
      if (p >= np) break;
      float acc[4];
      logits(a, qf[p], acc);
      float e0 = 0.f, e1 = 0.f;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (2 * t4 + j >= G) continue;
        if (w0 < nc[p]) e0 += ex2(acc[j] * scale2 - M[p][j]) * inv[p][j];
        if (w0 + 8 < nc[p]) e1 += ex2(acc[2 + j] * scale2 - M[p][j]) * inv[p][j];
      }
      e0 += __shfl_xor_sync(0xffffffffu, e0, 1);
      e0 += __shfl_xor_sync(0xffffffffu, e0, 2);
      e1 += __shfl_xor_sync(0xffffffffu, e1, 1);
      e1 += __shfl_xor_sync(0xffffffffu, e1, 2);
      if (t4 == 0) {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int w = w0 + 8 * hr;
          if (w >= nc[p]) continue;
          // window w overlaps blocks (w + 1) / 4 and, when w = 4 b + 3, also b = (w + 1) / 4 - 1
          const uint32_t bits = __float_as_uint(hr ? e1 : e0);
          const int b1 = (w + 1) >> 2;
          if (b1 < nbn) atomicMax(&pooled[p * nbn + b1], bits);
          if (((w + 1) & 3) == 0 && b1 >= 1) atomicMax(&pooled[p * nbn + b1 - 1], bits);
        }
      }
    }
  }
  __syncwarp();
  // a block with no complete window scores -inf, as in the decode step
  auto pooled_score = [&](int p, int b) {
    return (nc[p] >= 1 && 4 * b <= nc[p]) ? __uint_as_float(pooled[p * nbn + b]) : -INFINITY;
  };
  const int nbw = (nbn + 31) >> 5;
  uint32_t* qw = qword_sm[warp];
#pragma unroll
  for (int p = 0; p < PW; ++p) {
    if (p >= np) break;
    const int t = tw + p;
    const Geometry geo = geometry(t + 1, s.nw, s.sink);
    for (int w = lane; w < nbw; w += 32) qw[w] = 0u;
    __syncwarp();
    const int c0 = s.sink, c1 = geo.ws;  // candidates [c0, c1)
    unsigned long long thr = ~0ull;      // keys at or above it were taken by an earlier round
    for (int got = 0; got < kq; got += 32) {
      unsigned long long best = 0ull;    // below every real key (its block field is never 0)
      for (int bb = c0; bb < c1; bb += 32) {
        const int b = bb + lane;
        unsigned long long x = 0ull;
        if (b < c1) {
          x = rank_key(orderable(pooled_score(p, b)), b);
          if (x >= thr) x = 0ull;
        }
        best = warp_merge_top(best, warp_sort_desc(x));
      }
      if (best && lane < kq - got) {
        const int b = (int)(0xFFFFFFFFu - (uint32_t)best);
        atomicOr(&qw[b >> 5], 1u << (b & 31));
      }
      thr = __shfl_sync(0xffffffffu, best, 31);
      if (thr == 0ull) break;  // fewer candidates than k_q
    }
    __syncwarp();
    uint32_t* row = qsel + ((size_t)u * n + t) * nbw;
    for (int w = lane; w < nbw; w += 32) row[w] = qw[w];
    __syncwarp();
    if (t == n - 1)
      for (int b = lane; b < geo.nb; b += 32) s.sq_blk[(size_t)u * s.nb_max + b] = pooled_score(p, b);
  }
}

// ---------------------------------------------------------------- 2a'. the same on tcgen05
// A CTA takes PT consecutive positions of one unit (PT <= 128 / G, at most 32, fewer for long
// prompts: their pooled scores live in shared memory); Q holds their (position, head) rows as an
// M = 128 operand.  The unit's compressed keys stream through a TMA ring in tiles of 128 windows,
// twice.  Pass 1: S = Q K~^T (rows (position, head), columns windows) into tensor memory; one
// thread per row keeps its maximum and sum of exp over the windows complete at its position's T.
// Pass 2: S^T = K~ Q^T (rows windows, columns (position, head)); one thread per window forms, for
// each position, the group softmax summed over its heads (maxima and sums of pass 1 from shared
// memory) and max-pools it onto the blocks the window overlaps (shared-memory atomics).  Then each
// position's top k_q candidates, as in 2a.  Roles: warp 0 lane 0 issues the MMAs, warp 1 lane 0
// the loads, warps 4-7 the rows and windows; 256 tensor-memory columns (two 128-column buffers).
// Used for groups of up to four q heads per kv head, where its 128 rows hold 32 positions; with
// eight heads a CTA holds only 16 and the per-window pooling (one thread per window, every
// position) outweighs the MMAs it saves, so those groups take 2a.
constexpr int kQtMaxGroup = 4;
constexpr int kQtStages = 3;
constexpr int kQtThreads = 256;
constexpr int kQtTileBytes = 128 * 256;  // 128 windows x 128 dims bf16

__host__ __device__ inline int qt_positions(int G, int nbn) {
  const int by_rows = kTcRowsQ / G < 32 ? kTcRowsQ / G : 32;
  const int by_smem = 16384 / nbn;  // pooled scores: PT x nbn floats <= 64 KiB
  return by_rows < by_smem ? by_rows : (by_smem > 0 ? by_smem : 1);
}
__host__ __device__ inline size_t qt_smem_bytes(int PT, int nbn) {
  return 1024 + 32768 + (size_t)kQtStages * kQtTileBytes + (size_t)PT * nbn * 4 + 2 * 128 * 4 + 4 * kPfMaxWords * 4 + 32 * 4;
}

template <int G>
__global__ void __launch_bounds__(kQtThreads, 1)
    prefill_query_tc_kernel(const __grid_constant__ CUtensorMap tkt, LayerState s, const uint16_t* __restrict__ q,
                            uint32_t* __restrict__ qsel, int n, int nbn, int PT) {
  extern __shared__ unsigned char qsm_raw[];
  __shared__ __align__(8) uint64_t full[kQtStages], empty[kQtStages], s_full[2], s_free[2], stats_bar, pool_bar,
      drain;
  __shared__ uint32_t tbase;
  __shared__ int bad_flag;
  unsigned char* sm =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(qsm_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sQ = sm;                                     // [2 dim halves][128 rows][128 B]
  unsigned char* sT = sQ + 32768;                             // [stage][2 dim halves][128 windows][128 B]
  uint32_t* pooled = reinterpret_cast<uint32_t*>(sT + kQtStages * kQtTileBytes);  // [PT][nbn] float bits
  float* colM = reinterpret_cast<float*>(pooled + (size_t)PT * nbn);  // per (position, head) row
  float* colI = colM + 128;
  uint32_t* qw_all = reinterpret_cast<uint32_t*>(colI + 128);  // [4 warps][kPfMaxWords]
  int* ncp = reinterpret_cast<int*>(qw_all + 4 * kPfMaxWords); // windows complete at each position
  const int u = blockIdx.y, t0 = blockIdx.x * PT;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int np = min(PT, n - t0);
  const int kq = s.k_q;
  const long long lim = s.wait_limit;
  const float scale2 = s.scale * 1.4426950408889634f;  // logits in base 2
  if (tid == 0) {
    prefetch_tmap(&tkt);
    for (int i = 0; i < kQtStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 128);
    }
    mbar_init(&stats_bar, 128);
    mbar_init(&pool_bar, 128);
    mbar_init(&drain, 1);
    fence_mbar_init();
    bad_flag = 0;
  }
  if (warp == 0) tc::alloc(&tbase, 256);
  pdl_wait();  // the bulk append wrote the compressed keys
  for (int i = tid; i < PT * nbn; i += kQtThreads) pooled[i] = 0u;  // +0.0f: group scores are non-negative
  if (tid < 32) ncp[tid] = tid < np ? geometry(t0 + tid + 1, s.nw, s.sink).nc : 0;
  // Q rows (position p, head h) in the 128-byte swizzle; rows past PT G are zero
  for (int idx = tid; idx < 128 * 16; idx += kQtThreads) {
    const int r = idx >> 4, c = idx & 15, p = r / G, h = r % G;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (p < np) v = *reinterpret_cast<const uint4*>(q + (((size_t)u * G + h) * n + t0 + p) * kHeadDim + 8 * c);
    *reinterpret_cast<uint4*>(sQ + (c >> 3) * 16384 + r * 128 + ((((c & 7) ^ (r & 7)) & 7) << 4)) = v;
  }
  fence_proxy_async_smem();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tm = tbase;
  const int ncmax = geometry(t0 + np, s.nw, s.sink).nc;  // the last position's windows
  const int ntile = (ncmax + 127) / 128, nitem = 2 * ntile;  // pass 1 over the tiles, then pass 2
  const uint32_t sQa = smem_u32(sQ), sTa = smem_u32(sT);
  constexpr uint32_t idS = tc::f16_idesc(128, 128, 0);

  if (warp == 1 && lane == 0) {  // TMA producer
    int issued = 0;
    for (int i = 0; i < nitem; ++i) {
      const int st = i % kQtStages, tile = i % ntile;
      if (i >= kQtStages && !mbar_wait_bounded(&empty[st], (uint32_t)(((i / kQtStages) - 1) & 1), lim)) {
        atomicOr(&bad_flag, 1);
        break;
      }
      if (*(volatile int*)&bad_flag) break;
      const uint32_t dst = sTa + st * kQtTileBytes;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&full[st], kQtTileBytes);
      tma_load_3d(dst, &tkt, 0, 128 * tile, u, &full[st]);
      tma_load_3d(dst + 16384, &tkt, 64, 128 * tile, u, &full[st]);
      issued = i + 1;
    }
    for (int i = max(issued - kQtStages, 0); i < issued; ++i)
      mbar_wait_bounded(&full[i % kQtStages], (uint32_t)((i / kQtStages) & 1), kWaitCycles);
  } else if (warp == 0 && lane == 0) {  // MMA issuer
    bool ok = true;
    for (int i = 0; i < nitem && ok; ++i) {
      const int st = i % kQtStages, sb = i & 1;
      if (!mbar_wait_bounded(&full[st], (uint32_t)((i / kQtStages) & 1), lim) ||
          (i >= 2 && !mbar_wait_bounded(&s_free[sb], (uint32_t)(((i >> 1) - 1) & 1), lim))) {
        ok = false;
        break;
      }
      tc::fence_after();
      const uint32_t kb = sTa + st * kQtTileBytes;
      const bool pass1 = i < ntile;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {  // dims 16 kk .. 16 kk + 15: halves at +0 and +16384
        const uint32_t off = (uint32_t)(kk >> 2) * 16384 + (uint32_t)(kk & 3) * 32;
        const uint64_t dq = tc::sw128_desc(sQa + off), dk = tc::sw128_desc(kb + off);
        tc::mma_bf16(tm + 128 * sb, pass1 ? dq : dk, pass1 ? dk : dq, idS, kk > 0);
      }
      tc::commit(&s_full[sb]);
      tc::commit(&empty[st]);
    }
    if (!ok) atomicOr(&bad_flag, 1);
    tc::commit(&drain);
    mbar_wait_bounded(&drain, 0u, kWaitCycles);
  } else if (warp >= 4) {  // rows (pass 1) and windows (pass 2)
    const int r = tid - 128;
    const uint32_t trow = tm + ((uint32_t)(32 * (warp & 3)) << 16);
    const int pr = r / G;                      // pass 1: this row's position
    const bool row_ok = pr < np;
    const int ncr = row_ok ? ncp[pr] : 0;
    float m = -INFINITY, l = 0.f;
    bool good = true;
    for (int i = 0; i < nitem; ++i) {
      const int sb = i & 1, tile = i % ntile;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&s_full[sb], (uint32_t)((i >> 1) & 1), lim))) {
        good = false;
        break;
      }
      tc::fence_after();
      uint32_t v[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::ld32(trow + 128 * sb + 32 * c, v[c]);
      tc::wait_ld();
      tc::fence_before();
      mbar_arrive(&s_free[sb]);
      if (i < ntile) {  // pass 1: row (position, head) over this tile's 128 windows
        if (row_ok) {
          float mxp[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) mxp[k] = -INFINITY;
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            const float z = 128 * tile + c < ncr ? __uint_as_float(v[c >> 5][c & 31]) * scale2 : -INFINITY;
            mxp[c & 7] = fmaxf(mxp[c & 7], z);
          }
          const float mt = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                                 fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
          if (mt > -INFINITY) {
            const float mn = fmaxf(m, mt);
            float sp[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) sp[k] = 0.f;
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (128 * tile + c < ncr) sp[c & 7] += ex2(__uint_as_float(v[c >> 5][c & 31]) * scale2 - mn);
            const float st = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
            l = (mn > m ? l * ex2(m - mn) : l) + st;
            m = mn;
          }
        }
        if (i == ntile - 1) {  // the row's statistics for pass 2
          colM[r] = m;
          colI[r] = l > 0.f ? 1.f / l : 0.f;
          mbar_arrive(&stats_bar);
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(&stats_bar, 0u, lim))) {
            good = false;
            break;
          }
        }
      } else {  // pass 2: window w of the tile, columns (position, head)
        const int w = 128 * tile + r;
        float gs[128 / G < 32 ? 128 / G : 32];
#pragma unroll
        for (int pp = 0; pp < (128 / G < 32 ? 128 / G : 32); ++pp) gs[pp] = 0.f;
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const int pp = c / G;
          if (pp < (128 / G < 32 ? 128 / G : 32) && pp < np && w < ncp[pp])
            gs[pp] += ex2(__uint_as_float(v[c >> 5][c & 31]) * scale2 - colM[c]) * colI[c];
        }
        // window w overlaps blocks (w + 1) / 4 and, when w = 4 b + 3, also b = (w + 1) / 4 - 1
        const int b1 = (w + 1) >> 2;
#pragma unroll
        for (int pp = 0; pp < (128 / G < 32 ? 128 / G : 32); ++pp) {
          if (pp >= np || w >= ncp[pp]) continue;
          const uint32_t bits = __float_as_uint(gs[pp]);
          if (b1 < nbn) atomicMax(&pooled[pp * nbn + b1], bits);
          if (((w + 1) & 3) == 0 && b1 >= 1) atomicMax(&pooled[pp * nbn + b1 - 1], bits);
        }
      }
    }
    if (!good) atomicOr(&bad_flag, 1);
    // every window's contribution pooled: each position's top k_q candidates (warps 4-7 in turn)
    mbar_arrive(&pool_bar);
    const bool pooled_ok = __all_sync(0xffffffffu, mbar_wait_bounded(&pool_bar, 0u, lim));
    if (!pooled_ok) atomicOr(&bad_flag, 1);
    const int nbw = (nbn + 31) >> 5;
    uint32_t* qw = qw_all + (warp - 4) * kPfMaxWords;
    for (int pp = warp - 4; pp < np; pp += 4) {
      const int t = t0 + pp;
      const Geometry geo = geometry(t + 1, s.nw, s.sink);
      auto score = [&](int b) {
        return (geo.nc >= 1 && 4 * b <= geo.nc) ? __uint_as_float(pooled[pp * nbn + b]) : -INFINITY;
      };
      for (int w = lane; w < nbw; w += 32) qw[w] = 0u;
      __syncwarp();
      const int c0 = s.sink, c1 = geo.ws;  // candidates [c0, c1)
      unsigned long long thr = ~0ull;
      for (int got = 0; got < kq; got += 32) {
        unsigned long long best = 0ull;
        for (int bb = c0; bb < c1; bb += 32) {
          const int b = bb + lane;
          unsigned long long x = 0ull;
          if (b < c1) {
            x = rank_key(orderable(score(b)), b);
            if (x >= thr) x = 0ull;
          }
          best = warp_merge_top(best, warp_sort_desc(x));
        }
        if (best && lane < kq - got) {
          const int b = (int)(0xFFFFFFFFu - (uint32_t)best);
          atomicOr(&qw[b >> 5], 1u << (b & 31));
        }
        thr = __shfl_sync(0xffffffffu, best, 31);
        if (thr == 0ull) break;
      }
      __syncwarp();
      uint32_t* row = qsel + ((size_t)u * n + t) * nbw;
      for (int w = lane; w < nbw; w += 32) row[w] = (*(volatile int*)&bad_flag) ? 0u : qw[w];
      __syncwarp();
      if (t == n - 1)
        for (int b = lane; b < geo.nb; b += 32) s.sq_blk[(size_t)u * s.nb_max + b] = score(b);
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (tid == 0 && bad_flag) atomicOr(s.err, kErrTimeout);
  if (warp == 0) tc::dealloc(tm, 256);
}

// ---------------------------------------------------------------- 2b. the walk over the positions
// One warp per unit makes the stateful part of every position's selection, in order: the k_e
// query-agnostic picks among the candidates never dropped before and the sticky eviction
// update (with the locality counters against the previous selection).  Every
// candidate a selection leaves out is dropped for good, so the candidates still eligible are the
// last selection's never-dropped blocks plus the blocks that have just become candidates; the warp
// keeps them in a list ordered by (pooled s^e, then lower block), and a position's picks are the
// list's first k_e entries outside its query-aware picks.  Selections are bitmaps over the blocks.
// A position's work is one dependent chain of a single warp, so the loops run over the list
// entries and bitmap words the configuration needs (KS entries and NW words per lane).
constexpr int kWalkWarps = 4;
constexpr int kWalkMaxSlots = 9;  // list entries per lane: k_q + k_e + 1 <= 288

__host__ __device__ inline size_t walk_warp_bytes(int nbn) {
  const int nbw = (nbn + 31) / 32;
  return (size_t)32 * kWalkMaxSlots * 8 + 4 * (size_t)nbw * 4;
}

__device__ __forceinline__ uint32_t range_bits(int w, int lo, int hi) {  // bits of [lo, hi) in word w
  const int a = max(lo - 32 * w, 0), b = min(hi - 32 * w, 32);
  if (a >= b) return 0u;
  const uint32_t top = b == 32 ? 0xFFFFFFFFu : ((1u << b) - 1u);
  return top & ~((1u << a) - 1u);
}

__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// grid ceil(U / 4), 128 threads; dynamic shared memory 4 x walk_warp_bytes(nbn).  qsel: the
// query-aware picks of 2a, esel: the query-agnostic picks this kernel makes, both [U][n][nbw]
// bitmap words.  The list's blocks are also kept as a bitmap (lb): after a position's step the
// list holds exactly the never-dropped blocks of D, so D = Q | lb and E = lb & ~Q without
// touching the picks one by one.
// KS: list entries per lane (k_q + k_e + 1 <= 32 KS); NW: bitmap words per lane (nbn <= 1024 NW).
template <int KS, int NW>
__global__ void __launch_bounds__(kWalkWarps * 32)
    prefill_walk_kernel(LayerState s, const uint32_t* __restrict__ qsel, uint32_t* __restrict__ esel, int n,
                        int nbn) {
  extern __shared__ __align__(16) unsigned char wsm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x * kWalkWarps + warp;
  pdl_wait();  // the query-aware picks, and the bulk append's pooled eviction scores
  if (u >= s.U) return;  // no CTA-wide barrier follows
  const int nbw = (nbn + 31) / 32;
  unsigned char* base = wsm + (size_t)warp * walk_warp_bytes(nbn);
  unsigned long long* Lk = reinterpret_cast<unsigned long long*>(base);  // the eligible list, descending keys
  uint32_t* ev = reinterpret_cast<uint32_t*>(base + 32 * kWalkMaxSlots * 8);
  uint32_t* sprev = ev + nbw;  // the previous selection
  uint32_t* qbm = sprev + nbw;  // this position's query-aware picks
  uint32_t* lb = qbm + nbw;     // the list's blocks
  const int ke = s.k_e, cap = s.cap, sink = s.sink;
  const unsigned int lt = (1u << lane) - 1u;
  // an empty layer: nothing dropped or selected
  for (int w = lane; w < nbw; w += 32) ev[w] = sprev[w] = qbm[w] = lb[w] = 0u;
  __syncwarp();
  const float* se_blk = s.se_blk + (size_t)u * s.nb_max;
  const float* se_win = s.se_win + (size_t)u * s.nc_max;
  // list key of candidate b at T: its pooled s^e over the windows complete at T (only the last
  // two blocks can still change), then the lower block
  auto se_key = [&](int b, const Geometry& g) {
    float v;
    if (b >= g.nb - 2) {
      v = -INFINITY;
      for (int i = max(4 * b - 1, 0); i <= min(4 * b + 3, g.nc - 1); ++i) v = fmaxf(v, se_win[i]);
    } else {
      v = se_blk[b];
    }
    return rank_key(orderable(v), b);
  };
  int nL = 0;
  auto l_insert = [&](unsigned long long key) {  // at its place in the descending list
    int c = 0;
#pragma unroll
    for (int i = 0; i < KS; ++i) c += (lane + 32 * i < nL && Lk[lane + 32 * i] > key) ? 1 : 0;
    c = warp_sum(c);
    unsigned long long v[KS];
#pragma unroll
    for (int i = 0; i < KS; ++i) {
      const int j = lane + 32 * i;
      v[i] = (j >= c && j < nL) ? Lk[j] : 0ull;
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < KS; ++i) {
      const int j = lane + 32 * i;
      if (j >= c && j < nL && j + 1 < 32 * KS) Lk[j + 1] = v[i];
    }
    if (lane == 0 && c < 32 * KS) {
      Lk[c] = key;
      const int b = (int)(0xFFFFFFFFu - (uint32_t)key);
      lb[b >> 5] |= 1u << (b & 31);
    }
    __syncwarp();
    nL = min(nL + 1, 32 * KS);
  };
  // removes the entries of blocks >= bmin (at most two: the last two blocks) and returns them
  auto l_remove_from = [&](int bmin, unsigned long long& o0, unsigned long long& o1) {
    int nout = 0, wpos = 0;
    unsigned long long v[KS];
#pragma unroll
    for (int i = 0; i < KS; ++i) v[i] = lane + 32 * i < nL ? Lk[lane + 32 * i] : 0ull;
    __syncwarp();
#pragma unroll
    for (int i = 0; i < KS; ++i) {
      const bool in = lane + 32 * i < nL;
      const bool late = in && (int)(0xFFFFFFFFu - (uint32_t)v[i]) >= bmin;
      const unsigned int kb = __ballot_sync(0xffffffffu, in && !late), lb_ = __ballot_sync(0xffffffffu, late);
      if (in && !late) Lk[wpos + __popc(kb & lt)] = v[i];
      for (unsigned int m = lb_; m; m &= m - 1u) {
        const unsigned long long x = __shfl_sync(0xffffffffu, v[i], __ffs(m) - 1);
        if (nout == 0) o0 = x;
        else if (nout == 1) o1 = x;
        ++nout;
      }
      wpos += __popc(kb);
    }
    __syncwarp();
    nL = wpos;
    return min(nout, 2);
  };
  uint32_t qn[NW];  // the next position's query-aware words, loaded a position ahead
  auto load_q = [&](int t) {
#pragma unroll
    for (int k = 0; k < NW; ++k) {
      const int w = lane + 32 * k;
      qn[k] = (t < n && w < nbw) ? qsel[((size_t)u * n + t) * nbw + w] : 0u;
    }
  };
  load_q(0);
  unsigned long long st_short = 0, st_gs = 0, st_gn = 0, st_gd = 0;
  uint32_t st_gmin = 0x7F800000u;  // +inf
  int ws_prev = sink;               // candidates so far: [sink, ws_prev)
  int nS_prev = 0, nS = 0, nD = 0, nDnew = 0;
  uint32_t Sw[NW];
  Geometry geo = geometry(1, s.nw, s.sink);
  for (int t = 0; t < n; ++t) {
    geo = geometry(t + 1, s.nw, s.sink);
    const int nbwT = (geo.nb + 31) >> 5;
    uint32_t qc[NW];
#pragma unroll
    for (int k = 0; k < NW; ++k) {
      qc[k] = qn[k];
      if (lane + 32 * k < nbw) qbm[lane + 32 * k] = qc[k];
    }
    load_q(t + 1);  // in flight during this position
    // list keys that follow T (a window shorter than two blocks lets the last two blocks be
    // candidates), then the blocks that have just become candidates
    if (s.nw < 2 && nL > 0) {
      unsigned long long l0 = 0ull, l1 = 0ull;
      const int nlate = l_remove_from(geo.nb - 2, l0, l1);
      if (nlate > 0) l_insert(se_key((int)(0xFFFFFFFFu - (uint32_t)l0), geo));
      if (nlate > 1) l_insert(se_key((int)(0xFFFFFFFFu - (uint32_t)l1), geo));
    }
    for (int b = max(sink, ws_prev); b < geo.ws; ++b) l_insert(se_key(b, geo));
    ws_prev = max(ws_prev, geo.ws);
    __syncwarp();  // query-aware words visible to every lane
    // E: the list's first k_e entries outside Q; the other entries outside Q are dropped for good
    // (out of the list, its bitmap and the eligible set)
    int nElig = 0;
    unsigned long long v[KS];
    bool drop[KS];
    unsigned int anyd = 0u;
#pragma unroll
    for (int i = 0; i < KS; ++i) {
      const bool in = lane + 32 * i < nL;
      v[i] = in ? Lk[lane + 32 * i] : 0ull;
      const int b = (int)(0xFFFFFFFFu - (uint32_t)v[i]);
      const bool inQ = in && ((qbm[b >> 5] >> (b & 31)) & 1u);
      const bool elig = in && !inQ;
      const unsigned int eb = __ballot_sync(0xffffffffu, elig);
      drop[i] = elig && nElig + __popc(eb & lt) >= ke;
      nElig += __popc(eb);
      if (drop[i]) {
        atomicOr(&ev[b >> 5], 1u << (b & 31));
        atomicAnd(&lb[b >> 5], ~(1u << (b & 31)));
      }
      anyd |= __ballot_sync(0xffffffffu, drop[i]);
    }
    const int nE = min(ke, nElig);
    if (anyd) {  // the list keeps D's never-dropped blocks, in order
      __syncwarp();
      int wpos = 0;
#pragma unroll
      for (int i = 0; i < KS; ++i) {
        const bool keep = lane + 32 * i < nL && !drop[i];
        const unsigned int kb = __ballot_sync(0xffffffffu, keep);
        if (keep) Lk[wpos + __popc(kb & lt)] = v[i];
        wpos += __popc(kb);
      }
      nL = wpos;
    }
    __syncwarp();
    // S = sink + D + window per word, D = Q | the list's blocks; the blocks of D new to S (for the
    // locality counters); this position's query-agnostic words to the caller
    int cnt = 0;  // popc(D) | popc(D & new) << 10 (each at most 256)
    uint32_t* erow = esel + ((size_t)u * n + t) * nbw;
#pragma unroll
    for (int k = 0; k < NW; ++k) {
      const int w = lane + 32 * k;
      Sw[k] = 0u;
      if (w >= nbw) continue;
      const uint32_t L = lb[w];
      erow[w] = L & ~qc[k];
      if (w >= nbwT) continue;
      const uint32_t D = qc[k] | L;
      const uint32_t sw = D | range_bits(w, 0, geo.ns) | range_bits(w, geo.ws, geo.nb);
      Sw[k] = sw;
      cnt += __popc(D) | (__popc(D & ~sprev[w]) << 10);
    }
    cnt = warp_sum(cnt);
    nD = cnt & 1023;
    nDnew = (cnt >> 10) & 1023;
    nS = geo.ns + nD + (geo.nb - geo.ws);
    if (nS > cap && lane == 0) atomicOr(s.err, kErrBounds);  // cannot happen when cap = sink + window + k_q + k_e
    // the decode step's counters
    if (nE < ke) ++st_short;
    if (nS_prev > 0 && nD > 0) {  // some block was cached before
      ++st_gs;
      st_gn += nD - nDnew;
      st_gd += nD;
      st_gmin = min(st_gmin, __float_as_uint((float)(nD - nDnew) / (float)nD));
    }
    nS_prev = nS;
    // this selection is the next position's previous one (the last position's previous one
    // stays, for the fetched marks below)
    if (t + 1 < n) {
#pragma unroll
      for (int k = 0; k < NW; ++k)
        if (lane + 32 * k < nbwT) sprev[lane + 32 * k] = Sw[k];
    }
    __syncwarp();
  }
  // the unit's state after the prompt: the last selection with its kinds; the cache holds exactly
  // that selection, its i-th block in slot i (every block of it is written from the prompt next,
  // so nothing else is worth keeping), each slot marked as serving the selection at T = n; nothing
  // is left to fetch; the eviction bitmap
  int32_t* sel = s.sel + (size_t)u * cap;
  int32_t* kind = s.sel_kind + (size_t)u * cap;
  int32_t* sslot = s.sel_slot + (size_t)u * cap;
  int32_t* snew = s.sel_new + (size_t)u * cap;
  int32_t* b2s = s.blk2slot + (size_t)u * s.nb_max;
  const int nSw = min(nS, cap);
  for (int b = lane; b < nbn; b += 32) b2s[b] = -1;
  __syncwarp();
  {
    int pos = 0;
    const int nbwT = (geo.nb + 31) >> 5;
    for (int w = 0; w < nbwT; ++w) {
      const uint32_t mine = (NW > 1 && (w >> 5) == 1) ? Sw[NW - 1] : Sw[0];
      const uint32_t sw = __shfl_sync(0xffffffffu, mine, w & 31);
      if ((sw >> lane) & 1u) {
        const int p = pos + __popc(sw & lt), b = 32 * w + lane;
        if (p < nSw) {
          sel[p] = b;
          kind[p] = b < geo.ns ? 0 : b >= geo.ws ? 1 : ((qbm[w] >> lane) & 1u) ? 2 : 3;
          sslot[p] = p;
          snew[p] = 0;
          b2s[b] = p;
        }
      }
      pos += __popc(sw);
    }
  }
  for (int i = nSw + lane; i < cap; i += 32) {
    sel[i] = -1;
    kind[i] = -1;
    sslot[i] = -1;
    snew[i] = 0;
  }
  __syncwarp();  // the selection list above, read back by other lanes
  for (int i = lane; i < s.cslots; i += 32) {
    s.slot_blk[(size_t)u * s.cslots + i] = i < nSw ? sel[i] : -1;
    s.last_used[(size_t)u * s.cslots + i] = i < nSw ? n : -1;
  }
  if (lane == 0) {
    s.n_sel[u] = nSw;
    s.n_fetch[u] = 0;
    s.gamma[2 * u] = nD - nDnew;
    s.gamma[2 * u + 1] = nD;
  }
  for (int w = lane; w < s.ev_words; w += 32) s.evicted[(size_t)u * s.ev_words + w] = w < nbw ? ev[w] : 0u;
  if (lane == 0) {
    atomicAdd(&s.stats->selections, (unsigned long long)n);
    atomicAdd(&s.stats->short_selections, st_short);
    if (st_gs) {
      atomicAdd(&s.stats->gamma_samples, st_gs);
      atomicAdd(&s.stats->gamma_num, st_gn);
      atomicAdd(&s.stats->gamma_den, st_gd);
      atomicMin(&s.stats->gamma_min_bits, st_gmin);
    }
  }
}

// ---------------------------------------------------------------- 3. cache refresh
// grid (cap, U), 256 threads: slot `slot` of unit u receives its block from the prompt's K/V
// (rows past the prompt zero); after the prompt only the first |S| <= cap slots hold blocks.
__global__ void __launch_bounds__(256) prefill_refresh_kernel(LayerState s, const uint16_t* __restrict__ k,
                                                              const uint16_t* __restrict__ v, int n) {
  const int slot = blockIdx.x, u = blockIdx.y;
  pdl_wait();
  const int b = s.slot_blk[(size_t)u * s.cslots + slot];
  if (b < 0 || b * kBlock >= n) return;
  uint16_t* dst = s.cache + ((size_t)u * s.cslots + slot) * 2 * kBlockElems;
  for (int idx = threadIdx.x; idx < 2 * kBlock * 16; idx += blockDim.x) {
    const int kv = idx >> 10, r = (idx >> 4) & (kBlock - 1), c = idx & 15;
    const int tok = kBlock * b + r;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (tok < n) val = *reinterpret_cast<const uint4*>((kv ? v : k) + ((size_t)u * n + tok) * kHeadDim + 8 * c);
    *reinterpret_cast<uint4*>(dst + (size_t)kv * kBlockElems + r * kHeadDim + 8 * c) = val;
  }
}

// ---------------------------------------------------------------- 4. attention of every position (tcgen05)
// A CTA takes PT = 128 / G consecutive positions of one unit: its M = 128 rows are (position, q
// head) pairs, row r = p G + h (rows past PT G or past the prompt are padding).  It streams the
// union of the positions' selections block by block (TMA ring of K and V, 128-byte swizzle):
//   S_b = Q K_b^T (M 128, N 64 tokens, K 128 dims) into tensor memory (two buffers);
//   two threads per row (32 scores each) mask the block if the row's position did not select it
//   (and the tail tokens past the position), agree on the block maximum, and write the
//   probabilities exp2(z - m_ref) as bf16 to shared memory (two buffers), each adding its half to
//   its part of the row's sum;
//   O += P_b V_b (M 128, N 128 dims, K 64 tokens; V as an MN-major operand whose two 64-dim halves
//   are 16 KiB apart) accumulates in tensor memory across blocks.
// m_ref, the reference maximum of a row, is raised only when a block's maximum exceeds it by more
// than 8 (base 2): then the row's sum and its accumulated O (read and written back by the row's
// threads, once the previous product has completed) are scaled by exp2(old - new).  Probabilities
// stay below 2^8, and the output is O / sum with the same reference for both.
// Roles: warp 0 lane 0 issues the MMAs, warp 1 lane 0 the TMA loads, warps 4-11 own the rows, two
// threads per row (warps 4-7 columns 0-31, warps 8-11 columns 32-63 of a block, on the same
// tensor-memory lanes), exchanging their partial maxima through shared memory (an mbarrier per row
// quarter and block parity); warp 0 allocates and frees 256 tensor-memory columns.  Every
// wait is bounded; a CTA whose wait gives up flags a timeout, drains and writes NaN outputs.
constexpr int kTcRows = 128;
constexpr int kTcStages = 3;
constexpr int kTcThreads = 384;
constexpr uint32_t kTcCols = 256;  // S buffers at columns 0 and 64, O at 128
constexpr float kTcRescale = 8.f;  // base-2 growth of a row maximum that forces a rescale


__host__ __device__ inline int tc_positions(int G) { return kTcRows / G; }
__host__ __device__ inline size_t tc_smem_bytes(int G) {
  // 1024 alignment slack, Q 32 KiB, stages, two P buffers of 16 KiB, per-position block bitmaps,
  // union list, per-stage eviction scores
  return 1024 + 32768 + (size_t)kTcStages * kStageBytes + 2 * 16384 + (size_t)tc_positions(G) * kPfMaxWords * 4 +
         (size_t)kPfMaxWords * 32 * 2 + (size_t)kTcStages * kBlock * 4;
}

__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_attend_tc_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                             LayerState s, const uint16_t* __restrict__ q, uint16_t* __restrict__ out,
                             const uint32_t* __restrict__ qsel, const uint32_t* __restrict__ esel, int n) {
  extern __shared__ unsigned char tsm_raw[];
  __shared__ __align__(8) uint64_t full[kTcStages], empty[kTcStages], s_full[2], s_free[2], p_full[2], o_done[2],
      drain, xbar[4][2];
  __shared__ float xchg[2][2][kTcRows];  // [block parity][column half][row]: the partner's partial maximum
  __shared__ uint32_t tbase;
  __shared__ int n_union, bad_flag;
  unsigned char* sm =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(tsm_raw) + 1023) & ~uintptr_t(1023));
  const int G = s.G, PT = tc_positions(G);
  unsigned char* sQ = sm;                                   // [2 dim halves][128 rows][128 B]
  unsigned char* sStage = sQ + 32768;                       // [stage][dim half][K, V][64 tokens][128 B]
  unsigned char* sP = sStage + kTcStages * kStageBytes;     // [2][128 rows][64 tokens] bf16
  uint32_t* bm = reinterpret_cast<uint32_t*>(sP + 2 * 16384);  // [PT][kPfMaxWords]
  int16_t* ublk = reinterpret_cast<int16_t*>(bm + PT * kPfMaxWords);  // union, ascending
  float* sebuf = reinterpret_cast<float*>(ublk + kPfMaxWords * 32);   // [stage][64]
  const int u = blockIdx.y, t0 = blockIdx.x * PT;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int np = min(PT, n - t0);
  const int nb_last = (t0 + np + kBlock - 1) / kBlock;  // blocks of the last position's context
  const int nbw = (nb_last + 31) / 32;
  const int nbws = ((n + kBlock - 1) / kBlock + 31) / 32;  // words per position in qsel and esel
  const bool dma = s.dma_bias != 0;
  const long long lim = s.wait_limit;
  if (tid == 0) {
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 256);
      mbar_init(&p_full[i], 256);
      for (int qq = 0; qq < 4; ++qq) mbar_init(&xbar[qq][i], 64);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(&drain, 1);
    fence_mbar_init();
    bad_flag = 0;
  }
  if (warp == 0) tc::alloc(&tbase, kTcCols);
  pdl_wait();  // the selections, the prompt's q, K and V and (with the bias) the eviction scores
  // per-position selections: query-aware | query-agnostic | sink | window
  for (int idx = tid; idx < PT * kPfMaxWords; idx += kTcThreads) {
    const int p = idx / kPfMaxWords, w = idx % kPfMaxWords;
    uint32_t v = 0u;
    if (p < np && w < nbw) {
      const Geometry g = geometry(t0 + p + 1, s.nw, s.sink);
      const size_t o = ((size_t)u * n + t0 + p) * nbws + w;
      v = qsel[o] | esel[o] | range_bits(w, 0, g.ns) | range_bits(w, g.ws, g.nb);
    }
    bm[idx] = v;
  }
  // Q rows (position p, head h) in the 128-byte swizzle: row r, 16-byte chunk c of its dim half
  for (int idx = tid; idx < kTcRows * 16; idx += kTcThreads) {
    const int r = idx >> 4, c = idx & 15, p = r / G, h = r % G;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (p < np) v = *reinterpret_cast<const uint4*>(q + (((size_t)u * G + h) * n + t0 + p) * kHeadDim + 8 * c);
    *reinterpret_cast<uint4*>(sQ + (c >> 3) * 16384 + r * 128 + ((((c & 7) ^ (r & 7)) & 7) << 4)) = v;
  }
  __syncthreads();
  if (warp == 2) {  // the union of the positions' selections, ascending
    int base = 0;
    for (int w0 = 0; w0 < nbw; w0 += 32) {
      const int w = w0 + lane;
      uint32_t uni = 0u;
      if (w < nbw)
        for (int p = 0; p < np; ++p) uni |= bm[p * kPfMaxWords + w];
      const int c = __popc(uni);
      const int incl = warp_incl_scan(c);
      int pos = base + incl - c;
      for (; uni; uni &= uni - 1u) ublk[pos++] = (int16_t)(32 * w + __ffs(uni) - 1);
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) n_union = base;
  }
  fence_proxy_async_smem();  // Q (generic stores) is read by the tensor core
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const int nu = n_union;
  const uint32_t tm = tbase;
  const uint32_t sQa = smem_u32(sQ), sSa = smem_u32(sStage), sPa = smem_u32(sP);
  constexpr uint32_t idS = tc::f16_idesc(128, 64, 0), idO = tc::f16_idesc(128, 128, 1);

  if (warp == 1 && lane == 0) {  // TMA producer
    int issued = 0;
    for (int j = 0; j < nu; ++j) {
      const int st = j % kTcStages;
      if (j >= kTcStages && !mbar_wait_bounded(&empty[st], (uint32_t)(((j / kTcStages) - 1) & 1), lim)) {
        atomicOr(&bad_flag, 1);
        break;
      }
      if (*(volatile int*)&bad_flag) break;
      const int b = ublk[j];
      const uint32_t dst = sSa + st * kStageBytes;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&full[st], kStageBytes + (dma ? kBlock * 4 : 0));
      tma_load_3d(dst, &tk, 0, kBlock * b, u, &full[st]);
      tma_load_3d(dst + 8192, &tv, 0, kBlock * b, u, &full[st]);
      tma_load_3d(dst + 16384, &tk, 64, kBlock * b, u, &full[st]);
      tma_load_3d(dst + 24576, &tv, 64, kBlock * b, u, &full[st]);
      if (dma)
        bulk_copy_g2s(smem_u32(sebuf + st * kBlock), s.se_tok + (size_t)u * s.se_stride + (size_t)kBlock * b,
                      kBlock * 4, &full[st]);
      issued = j + 1;
    }
    // the last loads have landed before the shared memory goes away (on the normal path the MMA
    // issuer has already waited for every one of them)
    for (int j = max(issued - kTcStages, 0); j < issued; ++j)
      mbar_wait_bounded(&full[j % kTcStages], (uint32_t)((j / kTcStages) & 1), kWaitCycles);
  } else if (warp == 0 && lane == 0) {  // MMA issuer
    auto issue_s = [&](int j) -> bool {  // S_j = Q K_j^T into buffer j & 1
      const int st = j % kTcStages, sb = j & 1;
      if (!mbar_wait_bounded(&full[st], (uint32_t)((j / kTcStages) & 1), lim)) return false;
      if (j >= 2 && !mbar_wait_bounded(&s_free[sb], (uint32_t)(((j >> 1) - 1) & 1), lim)) return false;
      tc::fence_after();
      const uint32_t kb = sSa + st * kStageBytes;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {  // dims 16 kk .. 16 kk + 15: K halves at +0 and +16384
        const uint32_t off = (uint32_t)(kk >> 2) * 16384 + (uint32_t)(kk & 3) * 32;
        tc::mma_bf16(tm + 64 * sb, tc::sw128_desc(sQa + off), tc::sw128_desc(kb + off), idS, kk > 0);
      }
      tc::commit(&s_full[sb]);
      return true;
    };
    bool ok = nu == 0 || issue_s(0);
    for (int j = 0; ok && j < nu; ++j) {
      if (j + 1 < nu && !issue_s(j + 1)) {
        ok = false;
        break;
      }
      const int pb = j & 1;
      if (!mbar_wait_bounded(&p_full[pb], (uint32_t)((j >> 1) & 1), lim)) {
        ok = false;
        break;
      }
      tc::fence_after();
      const uint32_t vb = sSa + (j % kTcStages) * kStageBytes + 8192;  // V halves at +8192 and +24576
      const uint32_t pa = sPa + pb * 16384;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)  // tokens 16 kk .. 16 kk + 15: 16 rows of V per step, all 128 dims
        tc::mma_bf16(tm + 128, tc::sw128_desc(pa + 32 * kk), tc::sw128_desc_mn(vb + 2048 * kk, 16384), idO,
                     j > 0 || kk > 0);
      tc::commit(&o_done[pb]);
      tc::commit(&empty[j % kTcStages]);
    }
    if (!ok) atomicOr(&bad_flag, 1);
    tc::commit(&drain);  // arrives once every MMA issued above has completed
    mbar_wait_bounded(&drain, 0u, kWaitCycles);
  } else if (warp >= 4) {  // two threads per row: warps 4-7 columns 0-31, warps 8-11 columns 32-63
    const int hf = (warp - 4) >> 2, qr = warp & 3;
    const int r = 32 * qr + lane, p = r / G, h = r % G, col0 = 32 * hf;
    const bool row_ok = p < np;
    const int t = t0 + p;
    const uint32_t trow = tm + ((uint32_t)(32 * qr) << 16);  // this warp's tensor-memory lanes
    const float sl2 = s.scale * 1.4426950408889634f;
    float mref = -INFINITY, l = 0.f;  // l: this thread's half of the row's sum
    bool started = false, good = true;
    // the partner thread (same row, other half) exchanges one value per block through shared
    // memory; an mbarrier per row quarter and block parity (bounded wait) orders the exchange
    auto exchange = [&](int j, float v, float& other) -> bool {
      xchg[j & 1][hf][r] = v;
      mbar_arrive(&xbar[qr][j & 1]);
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&xbar[qr][j & 1], (uint32_t)((j >> 1) & 1), lim))) return false;
      other = xchg[j & 1][1 - hf][r];
      return true;
    };
    for (int j = 0; j < nu; ++j) {
      const int sb = j & 1, st = j % kTcStages, b = ublk[j];
      // waits are decided for the whole warp: the tensor-memory accesses below are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&s_full[sb], (uint32_t)((j >> 1) & 1), lim))) {
        good = false;
        break;
      }
      tc::fence_after();
      uint32_t sv[32];
      tc::ld32(trow + 64 * sb + col0, sv);
      tc::wait_ld();
      tc::fence_before();
      mbar_arrive(&s_free[sb]);
      const bool act = row_ok && ((bm[p * kPfMaxWords + (b >> 5)] >> (b & 31)) & 1u);
      const int valid = min(t + 1 - kBlock * b, kBlock) - col0;  // tokens of this half in the position's context
      // scores in base 2 with the tail masked; eight independent partial maxima
      float z[32];
      float mxp[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mxp[k] = -INFINITY;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float v = __uint_as_float(sv[i]) * sl2;
        if (dma) v = fmaf(sebuf[st * kBlock + col0 + i], 1.4426950408889634f, v);
        z[i] = i < valid ? v : -INFINITY;
        mxp[i & 7] = fmaxf(mxp[i & 7], z[i]);
      }
      const float mh = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                             fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
      float mo;
      if (!exchange(j, mh, mo)) {
        good = false;
        break;
      }
      const float mx = act ? fmaxf(mh, mo) : -INFINITY;  // the same in both threads of the row
      // raise the reference maximum: at once for a row with nothing accumulated yet, else when it
      // grew by more than the threshold (the row's O scaled in tensor memory, warp by warp)
      float alpha = 1.f;
      if (act && mx > mref) {
        if (!started) {
          mref = mx;
        } else if (mx > mref + kTcRescale) {
          alpha = ex2(mref - mx);
          mref = mx;
        }
      }
      started = started || act;
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
        if (j >= 1 &&
            !__all_sync(0xffffffffu, mbar_wait_bounded(&o_done[(j - 1) & 1], (uint32_t)(((j - 1) >> 1) & 1), lim))) {
          good = false;
          break;
        }
        tc::fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) {  // this thread's 64 of the row's 128 output columns
          uint32_t ov[32];
          tc::ld32(trow + 128 + 64 * hf + 32 * c, ov);
          tc::wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
          tc::st32(trow + 128 + 64 * hf + 32 * c, ov);
        }
        tc::wait_st();
        tc::fence_before();
        l *= alpha;
      }
      uint32_t pk[16];  // bf16 pairs of this half's 32 probabilities (0 for a block the row did not select)
      if (act) {
        float sp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) sp[k] = 0.f;
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float e0 = ex2(z[i] - mref), e1 = ex2(z[i + 1] - mref);  // 0 for masked tokens
          sp[(i >> 1) & 7] += e0 + e1;
          pk[i >> 1] = pack_bf16x2(e0, e1);
        }
        l += ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = 0u;
      }
      // this half of the row's P into buffer j & 1 once the product two blocks back has read it
      const int pb = j & 1;
      if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait_bounded(&o_done[pb], (uint32_t)(((j >> 1) - 1) & 1), lim))) {
        good = false;
        break;
      }
      unsigned char* prow = sP + pb * 16384 + r * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(prow + ((((col0 >> 3) + c) ^ (r & 7)) << 4)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_proxy_async_smem();
      mbar_arrive(&p_full[pb]);
    }
    if (!good) atomicOr(&bad_flag, 1);
    // the row's sum from both halves; the last product has completed: O / sum for this half
    float lo = 0.f;
    if (!exchange(nu, l, lo)) {
      good = false;
      atomicOr(&bad_flag, 1);
    }
    const float lrow = l + lo;
    if (__all_sync(0xffffffffu, good) && nu > 0 &&
        !__all_sync(0xffffffffu, mbar_wait_bounded(&o_done[(nu - 1) & 1], (uint32_t)(((nu - 1) >> 1) & 1), lim))) {
      good = false;
      atomicOr(&bad_flag, 1);
    }
    tc::fence_after();
    float O[64];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint32_t ov[32];
      tc::ld32(trow + 128 + 64 * hf + 32 * c, ov);
      tc::wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) O[32 * c + i] = __uint_as_float(ov[i]);
    }
    const bool bad = *(volatile int*)&bad_flag != 0 || !good;
    if (row_ok) {
      uint16_t* orow = out + (((size_t)u * G + h) * n + t) * kHeadDim + 64 * hf;
      const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t w4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a0 = bad ? __int_as_float(0x7fc00000) : (nu > 0 ? O[8 * c + 2 * e] * inv : 0.f);
          const float a1 = bad ? __int_as_float(0x7fc00000) : (nu > 0 ? O[8 * c + 2 * e + 1] * inv : 0.f);
          w4[e] = pack_bf16x2(a0, a1);
        }
        reinterpret_cast<uint4*>(orow)[c] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
    }
  }
  // every MMA and every load has completed (the issuers waited for them above)
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (tid == 0 && bad_flag) atomicOr(s.err, kErrTimeout);
  if (warp == 0) tc::dealloc(tm, kTcCols);
}

// ---------------------------------------------------------------- host side
// prompts of up to 65,536 tokens (1,024 blocks): four positions per query-aware warp and one
// bitmap word per walk lane; longer ones two and two
static bool prefill_wide(int nbn) { return nbn > 1024; }
static size_t query_smem(int nbn, int pw) { return (size_t)kPqWarps * pw * nbn * sizeof(uint32_t); }
static size_t walk_smem(int nbn) { return kWalkWarps * walk_warp_bytes(nbn); }

int prefill_max_tokens() { return kPfMaxWords * 32 * kBlock; }

cudaError_t init_prefill() {
  const int nbn = kPfMaxWords * 32;
  cudaError_t e = cudaFuncSetAttribute(prefill_attend_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)tc_smem_bytes(1));
  const int qt_max = (int)qt_smem_bytes(32, 512);  // the largest PT x nbn (16384 floats)
#define NOSA_QT_ATTR(GG)                                                                                      \
  if (e == cudaSuccess)                                                                                       \
    e = cudaFuncSetAttribute(prefill_query_tc_kernel<GG>, cudaFuncAttributeMaxDynamicSharedMemorySize, qt_max);
  NOSA_QT_ATTR(1) NOSA_QT_ATTR(2) NOSA_QT_ATTR(3) NOSA_QT_ATTR(4)
#undef NOSA_QT_ATTR
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(prefill_query_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)query_smem(1024, 4));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(prefill_query_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)query_smem(nbn, 2));
  return e;  // the walk's shared memory (4 x walk_warp_bytes) stays under the default 48 KiB
}

cudaError_t launch_prefill(const LayerState& s, const CUtensorMap* tk, const CUtensorMap* tv, const CUtensorMap* tkt,
                           const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* out, uint32_t* qsel,
                           uint32_t* esel, int n, bool wide, cudaStream_t st) {
  const int nbn = (n + kBlock - 1) / kBlock;
  wide = wide || prefill_wide(nbn);
  cudaError_t e;
  if (s.G <= kQtMaxGroup) {  // tensor-core scores: 128 rows of (position, q head) per CTA
    const int qpt = qt_positions(s.G, nbn);
    // positions along x: the CTAs resident at once take consecutive positions of one unit and
    // share its compressed keys in L2
    const dim3 qgrid((n + qpt - 1) / qpt, s.U);
    const size_t qsm = qt_smem_bytes(qpt, nbn);
#define NOSA_QT(GG) \
  launch_ex(prefill_query_tc_kernel<GG>, qgrid, dim3(kQtThreads), qsm, st, true, 0, *tkt, s, q, qsel, n, nbn, qpt)
    switch (s.G) {
      case 1: e = NOSA_QT(1); break;
      case 2: e = NOSA_QT(2); break;
      case 3: e = NOSA_QT(3); break;
      default: e = NOSA_QT(4); break;
    }
#undef NOSA_QT
  } else {  // larger groups: one warp's positions with all their heads on mma.sync
    const int pw = wide ? 2 : 4;
    const dim3 qgrid((n + kPqWarps * pw - 1) / (kPqWarps * pw), s.U);
    e = pw == 4 ? launch_ex(prefill_query_kernel<4>, qgrid, dim3(kPqWarps * 32), query_smem(nbn, 4), st, true, 0, s,
                            q, qsel, n, nbn)
                : launch_ex(prefill_query_kernel<2>, qgrid, dim3(kPqWarps * 32), query_smem(nbn, 2), st, true, 0, s,
                            q, qsel, n, nbn);
  }
  if (e != cudaSuccess) return e;
  // list entries and bitmap words per lane: as few as the configuration allows
  const int need = s.k_q + s.k_e + 1;
  const int ks = need <= 32 ? 1 : need <= 64 ? 2 : need <= 96 ? 3 : need <= 128 ? 4 : kWalkMaxSlots;
  const bool nw1 = !wide;
  const dim3 wgrid((s.U + kWalkWarps - 1) / kWalkWarps), wblock(kWalkWarps * 32);
  const size_t wsm = walk_smem(nbn);
  const uint32_t* qs = qsel;
#define NOSA_WALK(KS, NW) launch_ex(prefill_walk_kernel<KS, NW>, wgrid, wblock, wsm, st, true, 0, s, qs, esel, n, nbn)
  switch (ks) {
    case 1: e = nw1 ? NOSA_WALK(1, 1) : NOSA_WALK(1, 2); break;
    case 2: e = nw1 ? NOSA_WALK(2, 1) : NOSA_WALK(2, 2); break;
    case 3: e = nw1 ? NOSA_WALK(3, 1) : NOSA_WALK(3, 2); break;
    case 4: e = nw1 ? NOSA_WALK(4, 1) : NOSA_WALK(4, 2); break;
    default: e = nw1 ? NOSA_WALK(kWalkMaxSlots, 1) : NOSA_WALK(kWalkMaxSlots, 2); break;
  }
#undef NOSA_WALK
  if (e != cudaSuccess) return e;
  e = launch_ex(prefill_refresh_kernel, dim3(s.cap, s.U), dim3(256), 0, st, true, 0, s, k, v, n);
  if (e != cudaSuccess) return e;
  const int pt = tc_positions(s.G);
  // positions along x, as above: neighbouring positions' selections overlap, so the CTAs resident at
  // once read the same unit's blocks and most of them come from L2
  return launch_ex(prefill_attend_tc_kernel, dim3((n + pt - 1) / pt, s.U), dim3(kTcThreads), tc_smem_bytes(s.G), st,
                   true, 0, *tk, *tv, s, q, out, qs, static_cast<const uint32_t*>(esel), n);
}

}  // namespace nosa
