// nosa_attend_noalloc: the split-K sparse attention over a caller-owned block
// cache, for callers that cannot allocate device memory.
//
// Some callers run where cudaMalloc is off limits: inside a memory pool they
// do not own, in a process whose allocator is being captured or audited, or
// in code paths that must not grow the device footprint after start-up.  This
// entry point needs no context and allocates nothing: the kernel's scratch (the
// per-chunk partial results, the merge tickets and the context length) lives in
// one file-scope __device__ array of fixed size, which every GPU that loads
// this library keeps until the process exits.  The caller passes every input
// and output buffer.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "host.h"

namespace {

using namespace nosa;

constexpr int kNoAllocMaxUnits = 1024;
constexpr int kNoAllocMaxPartials = 2048;  // (unit, chunk) pairs
constexpr size_t kTicketsOff = 256;
constexpr size_t kPartialsOff = kTicketsOff + 2 * kNoAllocMaxUnits * sizeof(unsigned int) + 256;
constexpr size_t kScratchBytes = kPartialsOff + (size_t)kNoAllocMaxPartials * kMaxGroup * kPartStride * sizeof(float);

// [0]: context length, [4]: device error word (used when the caller passes none),
// [256...]: tickets, then partials.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
unsigned char* g_scratch_ptr[kMaxDevices] = {};

__global__ void noalloc_prepare_kernel(unsigned char* scratch, int* err, int T, int units) {
  int* hdr = reinterpret_cast<int*>(scratch);
  unsigned int* tickets = reinterpret_cast<unsigned int*>(scratch + kTicketsOff);
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i == 0) {
    hdr[0] = T;
    *err = 0;  // the error word this call reports into starts clear
  }
  if (i < 2 * units) tickets[i] = 0;  // merge tickets start at zero on every call
}

// Per-device set-up: the scratch address (host code must not use the symbol
// itself) and the attend kernel's shared-memory limit.  Runs once per device.
nosa_status scratch_for_current_device(unsigned char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return NOSA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return NOSA_ERR_CUDA;
    }
    if (init_attend() != cudaSuccess) {
      (void)cudaGetLastError();
      return NOSA_ERR_CUDA;
    }
    g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_scratch_ptr[dev];
  return NOSA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

}  // namespace

extern "C" nosa_status nosa_attend_noalloc(const uint16_t* q, const uint16_t* cache, const int32_t* sel,
                                           const int32_t* sel_slot, const int32_t* n_sel, int units, int group,
                                           int cache_slots, int context_len, float softmax_scale, uint16_t* out,
                                           int32_t* err_out, void* stream) {
  if (!q || !cache || !sel || !sel_slot || !n_sel || !out) return NOSA_ERR_INVALID_ARG;
  if (units < 1 || group < 1 || group > kMaxGroup || cache_slots < 1 || cache_slots > 256 || context_len < 1 ||
      !(softmax_scale >= 0.f))
    return NOSA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(cache) % 16) return NOSA_ERR_INVALID_ARG;  // TMA base alignment
  if (units > kNoAllocMaxUnits) return NOSA_ERR_CAPACITY;
  int num_sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return NOSA_ERR_CUDA;
  }
  if (reinterpret_cast<uintptr_t>(err_out) % 4) return NOSA_ERR_INVALID_ARG;
  // split-K chunking as in a context, widened until the partials fit the fixed scratch
  int bpc = (int)(((long long)units * cache_slots + 2ll * num_sms - 1) / (2ll * num_sms));
  bpc = std::min(std::max(bpc, 1), kMaxBlocksPerCta);
  while (bpc < kMaxBlocksPerCta && (long long)units * ((cache_slots + bpc - 1) / bpc) > kNoAllocMaxPartials) ++bpc;
  const int chunks = (cache_slots + bpc - 1) / bpc;
  if ((long long)units * chunks > kNoAllocMaxPartials) return NOSA_ERR_CAPACITY;

  unsigned char* scratch = nullptr;
  nosa_status st = scratch_for_current_device(&scratch);
  if (st != NOSA_OK) return st;
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return NOSA_ERR_CUDA;
  CUtensorMap tmap;
  cuuint64_t dims[4] = {(cuuint64_t)kHeadDim, (cuuint64_t)kBlock, 2, (cuuint64_t)units * cache_slots};
  cuuint64_t strides[3] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)kBlockElems * 2, (cuuint64_t)kBlockBytes};
  cuuint32_t box[4] = {64, (cuuint32_t)kBlock, 2, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  if (enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(cache), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return NOSA_ERR_INVALID_ARG;

  LayerState s{};
  s.layer = 0;
  s.U = units;
  s.G = group;
  s.Hkv = 1;
  s.cap = cache_slots;
  s.cslots = cache_slots;
  s.nw = 0;
  s.sink = 0;
  s.unit_base = 0;
  s.scale = softmax_scale > 0.f ? softmax_scale : 1.f / sqrtf((float)kHeadDim);
  s.T = reinterpret_cast<int*>(scratch);
  s.err = err_out ? reinterpret_cast<int*>(err_out) : reinterpret_cast<int*>(scratch) + 1;
  s.tickets = reinterpret_cast<unsigned int*>(scratch + kTicketsOff);
  s.apart = reinterpret_cast<float*>(scratch + kPartialsOff);
  s.sel = const_cast<int32_t*>(sel);
  s.sel_slot = const_cast<int32_t*>(sel_slot);
  s.n_sel = const_cast<int32_t*>(n_sel);
  s.attend_chunks = chunks;
  s.attend_mode = 0;  // merge by ticket in the fixed scratch
  s.wait_limit = kWaitCycles;
  s.dma_bias = 0;  // no eviction scores here: plain attention
  s.attend_blocks_per_cta = bpc;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  noalloc_prepare_kernel<<<(2 * units + 255) / 256, 256, 0, cs>>>(scratch, s.err, context_len, units);
  if (cudaGetLastError() != cudaSuccess) return NOSA_ERR_CUDA;
  if (launch_attend(s, &tmap, q, out, 0, false, cs) != cudaSuccess) {
    (void)cudaGetLastError();
    return NOSA_ERR_CUDA;
  }
  return NOSA_OK;
}
