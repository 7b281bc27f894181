// a1 append: new K/V into the pinned host store (UVA stores) and into the
// block-cache slot when the block is resident; per-token eviction score
// s^e = softplus(v W1) W2 (NOSA explainer eq. 4; wiki "How NOSA works": the
// DMA-style eviction head, ranked pre-exponential); every 16th token a new
// compressed key K~_i = bf16(mean of 32 keys) (NOSA-1B blog, key compressor:
// kernel 32, stride 16) and the window mean of s^e, max-pooled onto the
// 64-token blocks the window overlaps (explainer eq. 5-6).
#include "append_core.cuh"
#include "host.h"

namespace nosa {

// ---------------------------------------------------------------- one token per unit
// grid: U CTAs (one per unit), 256 threads.
constexpr int kAppendThreads = 256;

__global__ void __launch_bounds__(kAppendThreads) append_one_kernel(LayerState s, const uint16_t* __restrict__ knew,
                                                                    const uint16_t* __restrict__ vnew) {
  const int u = blockIdx.x, tid = threadIdx.x;
  // k_new and v_new may come from the previous kernel: wait before reading them
  pdl_wait();
  pdl_launch_dependents();  // the selector may start its own prologue
  const int p = *s.T;  // position of the new token (all CTAs read it before any ticket)
  if (p >= s.T_max) {
    if (tid == 0 && u == 0) atomicOr(s.err, kErrCapacity);
    return;  // every CTA sees the same p: nobody takes a ticket, T is unchanged
  }
  append_token<kAppendThreads>(s, u, p, knew, vnew, true);
  // the last CTA to finish advances the layer's context length
  if (tid == 0) {
    unsigned int* tk = s.tickets + 3 * s.U;
    const unsigned int t = atomicAdd(tk, 1u);
    if (t == gridDim.x - 1) {
      *tk = 0;
      *s.T = p + 1;
    }
  }
}

// ---------------------------------------------------------------- bulk context load
// B1: per (32-token tile, unit): host store (+ resident slots) and per-token s^e.
__global__ void __launch_bounds__(256) append_bulk_tokens_kernel(LayerState s, const uint16_t* __restrict__ k,
                                                                 const uint16_t* __restrict__ v, int T_old, int n) {
  extern __shared__ float sm[];
  const int tok0 = blockIdx.x * 32, u = blockIdx.y, tid = threadIdx.x;
  const int ntok = min(32, n - tok0);
  const int g = u % s.Hkv;
  const int h = s.h;
  float* W1s = sm;                        // [d][h]
  float* vs = sm + kHeadDim * h;          // [32][129]
  const uint16_t* kbase = k + ((size_t)u * n + tok0) * kHeadDim;
  const uint16_t* vbase = v + ((size_t)u * n + tok0) * kHeadDim;
  for (int idx = tid; idx < ntok * 32; idx += blockDim.x) {
    const int t = idx >> 5, half = (idx >> 4) & 1, c8 = (idx & 15) * 8;
    const int p = T_old + tok0 + t, blk = p / kBlock, row = p % kBlock;
    const uint4 val = *reinterpret_cast<const uint4*>((half ? vbase : kbase) + (size_t)t * kHeadDim + c8);
    const size_t hoff = (((size_t)u * s.nb_max + blk) * 2 + half) * kBlockElems + (size_t)row * kHeadDim + c8;
    *reinterpret_cast<uint4*>(s.host_kv + hoff) = val;
    const int slot = s.blk2slot[(size_t)u * s.nb_max + blk];
    if (slot >= s.cslots) {
      atomicOr(s.err, kErrBounds);
    } else if (slot >= 0) {
      const size_t coff = (((size_t)u * s.cslots + slot) * 2 + half) * kBlockElems + (size_t)row * kHeadDim + c8;
      *reinterpret_cast<uint4*>(s.cache + coff) = val;
    }
  }
  const float* W1g = s.W1 + (size_t)g * kHeadDim * h;
  for (int i = tid; i < kHeadDim * h; i += blockDim.x) W1s[i] = W1g[i];
  for (int i = tid; i < 32 * kHeadDim; i += blockDim.x) {
    const int t = i / kHeadDim, c = i % kHeadDim;
    vs[t * (kHeadDim + 1) + c] = t < ntok ? bf16_to_float(vbase[(size_t)t * kHeadDim + c]) : 0.f;
  }
  __syncthreads();
  const int t = tid >> 3, sub = tid & 7;
  const float* W2 = s.W2 + (size_t)g * h;
  float part = 0.f;
  for (int m = sub; m < h; m += 8) {
    float acc = 0.f;
#pragma unroll 8
    for (int c = 0; c < kHeadDim; ++c) acc = fmaf(vs[t * (kHeadDim + 1) + c], W1s[c * h + m], acc);
    part = fmaf(softplus(acc), W2[m], part);
  }
  part += __shfl_xor_sync(0xffffffffu, part, 1);
  part += __shfl_xor_sync(0xffffffffu, part, 2);
  part += __shfl_xor_sync(0xffffffffu, part, 4);
  if (sub == 0 && t < ntok) s.se_tok[(size_t)u * s.se_stride + T_old + tok0 + t] = part;
}

// B2: per (new window, unit): compressed key and window mean of s^e.  Keys of
// tokens before T_old come from the ring of the last 32 keys, the rest from k.
__global__ void __launch_bounds__(128) append_bulk_windows_kernel(LayerState s, const uint16_t* __restrict__ k,
                                                                  int T_old, int n, int i0) {
  const int i = i0 + blockIdx.x, u = blockIdx.y, tid = threadIdx.x;
  double acc = 0.0;
  for (int r = 0; r < kCmpKernel; ++r) {
    const int j = kCmpStride * i + r;
    const uint16_t b = j >= T_old ? k[((size_t)u * n + (j - T_old)) * kHeadDim + tid]
                                  : s.kring[((size_t)u * 32 + (j & 31)) * kHeadDim + tid];
    acc += bf16_to_double(b);
  }
  s.kt[((size_t)u * s.nc_max + i) * kHeadDim + tid] = double_to_bf16_rne(acc / kCmpKernel);
  if (tid < 32) {
    double e = (double)s.se_tok[(size_t)u * s.se_stride + kCmpStride * i + tid];
    e = warp_sum(e);
    if (tid == 0) s.se_win[(size_t)u * s.nc_max + i] = (float)(e / kCmpKernel);
  }
}

// B3: per unit: re-pool s^e of the blocks touched by the new windows, refresh
// the key ring with the newest tokens, publish the new context length.
__global__ void __launch_bounds__(128) append_bulk_finish_kernel(LayerState s, const uint16_t* __restrict__ k,
                                                                 int T_old, int n, int i0, int i1) {
  const int u = blockIdx.x, tid = threadIdx.x;
  const int T_new = T_old + n;
  if (i1 >= i0) {
    const int nc = i1 + 1;
    const int b_lo = (kCmpStride * i0) / kBlock, b_hi = (kCmpStride * i1 + kCmpKernel - 1) / kBlock;
    for (int b = b_lo + tid; b <= b_hi; b += blockDim.x) {
      const int lo = max(4 * b - 1, 0), hi = min(4 * b + 3, nc - 1);
      float m = -INFINITY;
      for (int i = lo; i <= hi; ++i) m = fmaxf(m, s.se_win[(size_t)u * s.nc_max + i]);
      s.se_blk[(size_t)u * s.nb_max + b] = m;
    }
  }
  for (int j = max(T_old, T_new - 32); j < T_new; ++j)
    s.kring[((size_t)u * 32 + (j & 31)) * kHeadDim + tid] = k[((size_t)u * n + (j - T_old)) * kHeadDim + tid];
  if (u == 0 && tid == 0) *s.T = T_new;
}

cudaError_t launch_append_one(const LayerState& s, const uint16_t* k, const uint16_t* v, bool pdl, cudaStream_t st) {
  return launch_ex(append_one_kernel, dim3(s.U), dim3(kAppendThreads), 0, st, pdl, 0, s, k, v);
}

static size_t bulk_tokens_smem(const LayerState& s) {
  return (size_t)(kHeadDim * s.h + 32 * (kHeadDim + 1)) * sizeof(float);
}

cudaError_t init_append(const LayerState& s) {
  return cudaFuncSetAttribute(append_bulk_tokens_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)bulk_tokens_smem(s));
}

cudaError_t launch_append_bulk(const LayerState& s, const uint16_t* k, const uint16_t* v, int T_old, int n,
                               cudaStream_t st) {
  const size_t smem = bulk_tokens_smem(s);
  append_bulk_tokens_kernel<<<dim3((n + 31) / 32, s.U), 256, smem, st>>>(s, k, v, T_old, n);
  const int T_new = T_old + n;
  const int nc_old = T_old < kCmpKernel ? 0 : (T_old - kCmpKernel) / kCmpStride + 1;
  const int nc_new = T_new < kCmpKernel ? 0 : (T_new - kCmpKernel) / kCmpStride + 1;
  if (nc_new > nc_old) append_bulk_windows_kernel<<<dim3(nc_new - nc_old, s.U), 128, 0, st>>>(s, k, T_old, n, nc_old);
  append_bulk_finish_kernel<<<s.U, 128, 0, st>>>(s, k, T_old, n, nc_old, nc_new - 1);
  return cudaGetLastError();
}

}  // namespace nosa
