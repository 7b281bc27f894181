// Dense GQA decode attention over a device-resident KV cache: the full-attention
// comparator of the NOSA wiki's decode-throughput table (NOSA on NOSI against full
// attention engines at matched equivalent batch).  Every token of the context is
// attended: the block-sparse path with the selection replaced by all blocks.
//
// grid (chunks, units), 128 threads: CTA (c, u) runs the attention core over the
// contiguous blocks [c*bpc, (c+1)*bpc) of unit u (TMA ring, no host blocks), writes
// its (m, l, O) partial to the caller's scratch, and attend_merge_kernel combines
// the unit's partials.
#include <cudaTypedefs.h>

#include <algorithm>

#include "attend_core.cuh"
#include "host.h"

namespace nosa {

constexpr int kDenseStages = 3;
constexpr int kDenseMaxBlocksPerCta = 64;
constexpr size_t kDenseErrBytes = 256;  // the scratch starts with the device error word

__global__ void __launch_bounds__(kTeamThreads, 1)
    dense_attend_kernel(const __grid_constant__ CUtensorMap tmap, LayerState s, const uint16_t* __restrict__ q,
                        int T, int bpc) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[kDenseStages];
  __shared__ float wm[4][kMaxGroup], wl[4][kMaxGroup];
  __shared__ int s_blk[kDenseMaxBlocksPerCta], s_slot[kDenseMaxBlocksPerCta], s_new[kDenseMaxBlocksPerCta];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int chunk = blockIdx.x, u = blockIdx.y, tid = threadIdx.x, lane = tid & 31;
  const Geometry geo = geometry(T, 0, 0);
  const int b0 = chunk * bpc, n = max(min(bpc, geo.nb - b0), 0);
  for (int i = tid; i < n; i += blockDim.x) {
    s_blk[i] = b0 + i;
    s_slot[i] = b0 + i;  // the KV store holds block b of unit u at row u * cap + b
    s_new[i] = 0;
  }
  if (tid == 0) {
    prefetch_tmap(&tmap);
    for (int i = 0; i < kDenseStages; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  pdl_wait();  // q and the KV store may come from the previous kernel
  pdl_launch_dependents();
  uint32_t qb[8][2];
  load_q_frags(qb, q, u, s.G, lane);
  __syncthreads();
  WarpAcc A;
  A.init();
  attend_worker(&tmap, s, geo, u, qb, s_blk, s_slot, s_new, n, smem_u32(smem), bars, kDenseStages, nullptr,
                Team{0}, tid, A);
  __syncthreads();  // every copy has landed (or was drained): the stages can hold the warp partials
  float* wo = reinterpret_cast<float*>(smem);
  float* part0 = s.apart + ((size_t)u * s.attend_chunks + chunk) * kMaxGroup * kPartStride;
  cta_partial<4>(A, wm, wl, wo, s.G, [&](int h, int x, float M, float L, float O) {
    float* part = part0 + h * kPartStride;
    if (x == 0) {
      part[0] = M;
      part[1] = L;
    }
    part[2 + x] = O;
  });
}

// Blocks per CTA: about two CTAs per SM in total, at most kDenseMaxBlocksPerCta, and at
// most 256 chunks per unit (the merge kernel's limit).
static int dense_bpc(int units, int nb, int sms) {
  const long long want = ((long long)units * nb + 2ll * sms - 1) / (2ll * sms);
  const long long lo = std::max<long long>(want, (nb + 255) / 256);
  return (int)std::min<long long>(std::max<long long>(lo, 1), kDenseMaxBlocksPerCta);
}

static int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return sms;
}

size_t dense_scratch_bytes(int units, int context_len) {
  const int sms = device_sms();
  if (sms <= 0 || units < 1 || context_len < 1) return 0;
  const int nb = (context_len + kBlock - 1) / kBlock;
  const int chunks = (nb + dense_bpc(units, nb, sms) - 1) / dense_bpc(units, nb, sms);
  return kDenseErrBytes + (size_t)units * chunks * kMaxGroup * kPartStride * sizeof(float);
}

static PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      (void)cudaGetLastError();
  }
  return fn;
}

}  // namespace nosa

using namespace nosa;

extern "C" size_t nosa_dense_scratch_bytes(int units, int context_len) { return dense_scratch_bytes(units, context_len); }

extern "C" nosa_status nosa_dense_attend(const uint16_t* q, const uint16_t* kv, int units, int group, int max_blocks,
                                         int context_len, float softmax_scale, uint16_t* out, void* scratch,
                                         size_t scratch_bytes, void* stream) {
  if (!q || !kv || !out || !scratch) return NOSA_ERR_INVALID_ARG;
  if (units < 1 || group < 1 || group > kMaxGroup || context_len < 1 || max_blocks < 1 ||
      context_len > (long long)max_blocks * kBlock || context_len > 256 * kDenseMaxBlocksPerCta * kBlock ||
      !(softmax_scale >= 0.f))
    return NOSA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(kv) % 16 || reinterpret_cast<uintptr_t>(scratch) % 256) return NOSA_ERR_INVALID_ARG;
  if ((long long)units * max_blocks >= (1ll << 31)) return NOSA_ERR_INVALID_ARG;
  const int sms = device_sms();
  if (sms <= 0) return NOSA_ERR_CUDA;
  const int nb = (context_len + kBlock - 1) / kBlock;
  const int bpc = dense_bpc(units, nb, sms);
  const int chunks = (nb + bpc - 1) / bpc;
  if (scratch_bytes < dense_scratch_bytes(units, context_len)) return NOSA_ERR_CAPACITY;
  // kernel attributes (per device; cheap to set again)
  if (cudaFuncSetAttribute(dense_attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)(1024 + kDenseStages * kStageBytes)) != cudaSuccess) {
    (void)cudaGetLastError();
    return NOSA_ERR_CUDA;
  }
  PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
  if (!enc) return NOSA_ERR_CUDA;
  CUtensorMap tmap;
  cuuint64_t dims[4] = {(cuuint64_t)kHeadDim, (cuuint64_t)kBlock, 2, (cuuint64_t)units * max_blocks};
  cuuint64_t strides[3] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)kBlockElems * 2, (cuuint64_t)kBlockBytes};
  cuuint32_t box[4] = {64, (cuuint32_t)kBlock, 2, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  if (enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(kv), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return NOSA_ERR_INVALID_ARG;
  LayerState s{};
  s.U = units;
  s.G = group;
  s.Hkv = 1;
  s.cap = max_blocks;
  s.cslots = max_blocks;
  s.nb_max = max_blocks;
  s.unit_base = 0;
  s.scale = softmax_scale > 0.f ? softmax_scale : 1.f / sqrtf((float)kHeadDim);
  s.cache = const_cast<uint16_t*>(kv);
  s.err = reinterpret_cast<int*>(scratch);
  s.apart = reinterpret_cast<float*>(static_cast<unsigned char*>(scratch) + kDenseErrBytes);
  s.attend_chunks = chunks;
  s.wait_limit = kWaitCycles;
  s.dma_bias = 0;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (launch_ex(dense_attend_kernel, dim3(chunks, units), dim3(kTeamThreads), 1024 + kDenseStages * kStageBytes, cs,
                true, 0, tmap, s, q, context_len, bpc) != cudaSuccess) {
    (void)cudaGetLastError();
    return NOSA_ERR_CUDA;
  }
  if (launch_attend_merge(s, out, cs) != cudaSuccess) {
    (void)cudaGetLastError();
    return NOSA_ERR_CUDA;
  }
  return NOSA_OK;
}
