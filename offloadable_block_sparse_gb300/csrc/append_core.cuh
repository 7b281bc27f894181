// a1 append of one token per unit (NOSA explainer eq. 4; wiki "How NOSA works":
// the DMA-style eviction head, ranked pre-exponential; NOSA-1B blog, key
// compressor: kernel 32, stride 16; explainer eq. 5-6 for the pooling), shared
// by the append kernel and the fused decode kernel.
#pragma once

#include "nosa_internal.cuh"
#include "ptx.cuh"

namespace nosa {

// The compressed key of window wi = (p + 1 - 32) / 16, completed by the token at
// position p (key k_new): the exact float64 mean of the 32 keys (31 from the ring
// of the last 32 keys, then k_new), rounded once to bf16.  Threads 0..127 of the
// caller, one head dimension each.
__device__ __forceinline__ void window_key(const LayerState& s, int u, int p, int wi, const uint16_t* knew) {
  const int tid = threadIdx.x;
  if (tid >= kHeadDim) return;
  const uint16_t* rp = s.kring + (size_t)u * 32 * kHeadDim + tid;
  uint16_t ring[kCmpKernel - 1];
#pragma unroll
  for (int r = 0; r < kCmpKernel - 1; ++r) ring[r] = rp[((p - (kCmpKernel - 1) + r) & 31) * kHeadDim];
  double acc = bf16_to_double(knew[(size_t)u * kHeadDim + tid]);
#pragma unroll
  for (int r = 0; r < kCmpKernel - 1; ++r) acc += bf16_to_double(ring[r]);
  s.kt[((size_t)u * s.nc_max + wi) * kHeadDim + tid] = double_to_bf16_rne(acc / kCmpKernel);
}

// Appends the token at position p (< T_max) of unit u with kThreads (128 or 256) threads: the new K/V
// row into the host store (UVA stores) and into the block-cache slot when the block
// is resident, the key ring, s^e of the token, and on a window completion the
// window mean of s^e pooled into the blocks it overlaps, plus (write_kt) the
// window's compressed key.  The eviction-head matvec gives each thread one hidden
// unit and 128 (or, with 256 threads, half of the) input dims, whose W1 loads it
// issues back to back (one memory round trip rather than a dependent chain).
template <int kThreads>
__device__ __forceinline__ void append_token(const LayerState& s, int u, int p, const uint16_t* __restrict__ knew,
                                             const uint16_t* __restrict__ vnew, bool write_kt) {
  static_assert(kThreads == 128 || kThreads == 256, "one or two threads per hidden unit");
  constexpr int kPer = kHeadDim * kHeadDim / kThreads;  // input dims per thread: 128 or 64
  __shared__ float vf[kHeadDim];
  __shared__ float half_acc[2][kHeadDim];
  __shared__ float red[4];
  const int tid = threadIdx.x;
  const int blk = p / kBlock, row = p % kBlock;
  const int T = p + 1;
  const bool window_done = T >= kCmpKernel && (T - kCmpKernel) % kCmpStride == 0;
  const int wi = window_done ? (T - kCmpKernel) / kCmpStride : 0;  // window [16wi, 16wi+32) completes now
  const uint16_t* krow = knew + (size_t)u * kHeadDim;
  const uint16_t* vrow = vnew + (size_t)u * kHeadDim;
  const int g = u % s.Hkv;
  const float* W1 = s.W1 + (size_t)g * kHeadDim * s.h;
  const float* W2 = s.W2 + (size_t)g * s.h;
  const int mi = tid & (kHeadDim - 1), hf = tid >> 7;

  // ---- every load the step needs, issued together (one memory round trip)
  uint4 rowv = make_uint4(0, 0, 0, 0);
  int slot = -1;
  if (tid < 32) {
    rowv = *reinterpret_cast<const uint4*>(((tid >> 4) ? vrow : krow) + (tid & 15) * 8);
    slot = s.blk2slot[(size_t)u * s.nb_max + blk];
  }
  uint16_t kb = 0, vb = 0;
  float w2 = 0.f;
  if (tid < kHeadDim) {
    kb = krow[tid];
    vb = vrow[tid];
    w2 = W2[mi];
  }
  float w[kPer];
  {
    const float* wp = W1 + (size_t)(hf * kPer) * s.h + mi;
#pragma unroll
    for (int c = 0; c < kPer; ++c) w[c] = wp[(size_t)c * s.h];
  }
  float se_prev = 0.f, sb1 = 0.f, sb2 = 0.f;
  if (window_done) {
    if (tid < kCmpKernel - 1) se_prev = s.se_tok[(size_t)u * s.se_stride + p - (kCmpKernel - 1) + tid];
    if (tid == 0) {
      const float* sb = s.se_blk + (size_t)u * s.nb_max;
      sb1 = sb[(kCmpStride * wi) / kBlock];
      sb2 = sb[(kCmpStride * wi + kCmpKernel - 1) / kBlock];
    }
  }
  // the compressed key reads the ring before this token's key enters it
  if (window_done && write_kt) window_key(s, u, p, wi, knew);

  // ---- stores of the new token: host store (UVA), resident cache slot, key ring
  if (tid < 32) {
    const int half = tid >> 4, c8 = (tid & 15) * 8;
    const size_t hoff = (((size_t)u * s.nb_max + blk) * 2 + half) * kBlockElems + (size_t)row * kHeadDim + c8;
    *reinterpret_cast<uint4*>(s.host_kv + hoff) = rowv;  // store through the UVA alias of pinned memory
    if (slot >= s.cslots) {
      atomicOr(s.err, kErrBounds);
    } else if (slot >= 0) {
      const size_t coff = (((size_t)u * s.cslots + slot) * 2 + half) * kBlockElems + (size_t)row * kHeadDim + c8;
      *reinterpret_cast<uint4*>(s.cache + coff) = rowv;
    }
  }
  __syncthreads();  // the ring rows of the window key are read
  if (tid < kHeadDim) {
    s.kring[((size_t)u * 32 + (p & 31)) * kHeadDim + tid] = kb;
    vf[tid] = bf16_to_float(vb);
  }
  __syncthreads();

  // ---- eviction head: s^e = sum_m W2[m] softplus(sum_c v[c] W1[c][m]); two halves of c per m
  float part = 0.f;
  for (int m0 = 0; m0 < s.h; m0 += kHeadDim) {
    if (m0 > 0) {  // hidden sizes above 128: further column blocks
      const float* wp = W1 + (size_t)(hf * kPer) * s.h + m0 + mi;
#pragma unroll
      for (int c = 0; c < kPer; ++c) w[c] = wp[(size_t)c * s.h];
      if (tid < kHeadDim) w2 = W2[m0 + mi];
    }
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < kPer; ++c) acc = fmaf(vf[hf * kPer + c], w[c], acc);
    half_acc[hf][mi] = acc;
    __syncthreads();
    if (tid < kHeadDim) {
      const float hsum = kThreads == 256 ? half_acc[0][mi] + half_acc[1][mi] : half_acc[0][mi];
      part = fmaf(softplus(hsum), w2, part);
    }
    __syncthreads();
  }
  if (tid < kHeadDim) {
    part = warp_sum(part);
    if ((tid & 31) == 0) red[tid >> 5] = part;
  }
  __syncthreads();
  const float se = (red[0] + red[1]) + (red[2] + red[3]);
  if (tid == 0) s.se_tok[(size_t)u * s.se_stride + p] = se;

  // ---- a completed window: window mean of s^e, pooled onto the blocks it overlaps
  if (window_done && tid < 32) {
    double e = (double)(tid < kCmpKernel - 1 ? se_prev : se);
    e = warp_sum(e);
    if (tid == 0) {
      const float mean = (float)(e / kCmpKernel);
      s.se_win[(size_t)u * s.nc_max + wi] = mean;
      const int b1 = (kCmpStride * wi) / kBlock, b2 = (kCmpStride * wi + kCmpKernel - 1) / kBlock;
      float* sb = s.se_blk + (size_t)u * s.nb_max;
      sb[b1] = fmaxf(sb1, mean);
      if (b2 != b1) sb[b2] = fmaxf(sb2, mean);
    }
  }
  __syncthreads();
}

}  // namespace nosa
