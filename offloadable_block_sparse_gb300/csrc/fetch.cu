// a5 fetch: persistent UVA gather of newly selected blocks from the pinned host
// store into their cache slots (wiki "NOSI": a host-to-device kernel that reads
// CPU memory directly through Unified Virtual Addressing, block-wise 16 KiB
// transfers; SparDA summary, KV prefetch runtime: a small resident set of CTAs
// handles all copy work, CTA count traded against compute SMs).
//
// One work item is one block: its K and V chunks (2 x 16 KiB) are contiguous in
// both the host store and the slot.  Each thread moves 4 x 16 bytes per item; the
// CTA walks items item = blockIdx.x, += gridDim.x and keeps two items in flight: the
// loads of the next item are issued before the stores of the current one, so every
// CTA always has a host round trip under way.  Rows past the end of the partial tail
// block are written as zeros.  ahead = 1: the list comes from a forecast selection for
// T + 1 and may name the block the next token starts, which has no rows yet (all zeros
// here; the append writes its first row into the slot).
#include "host.h"
#include "ptx.cuh"

namespace nosa {

constexpr int kMaxGatherUnits = 4096;

__global__ void __launch_bounds__(kGatherThreads) gather_kernel(LayerState s, int ahead) {
  __shared__ int pref[kMaxGatherUnits + 1];
  __shared__ int scan_tmp[32];
  const int tid = threadIdx.x;
  const Geometry geo = geometry(*s.T, s.nw, s.sink);
  const int nb_sel = geometry(*s.T + ahead, s.nw, s.sink).nb;  // blocks of the selection's context
  // exclusive prefix of the per-unit fetch counts
  int carry = 0;
  for (int base = 0; base < s.U; base += blockDim.x) {
    const int uu = base + tid;
    const int v = uu < s.U ? s.n_fetch[uu] : 0;
    int tot;
    const int ex = block_scan_excl(v, scan_tmp, &tot);
    if (uu < s.U) pref[uu] = carry + ex;
    carry += tot;
  }
  if (tid == 0) pref[s.U] = carry;
  __syncthreads();
  const int total = carry;
  constexpr int kVec = kBlockBytes / 16 / kGatherThreads;  // 16-byte vectors per thread per block (4)
  struct Job {
    const uint4* src;
    uint4* dst;
    int rows;  // rows of the block that exist; -1: nothing to copy
  };
  auto job = [&](int item) -> Job {
    Job j{nullptr, nullptr, -1};
    if (item >= total) return j;
    int lo = 0, hi = s.U - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pref[mid] <= item) lo = mid;
      else hi = mid - 1;
    }
    const int u = lo, e = item - pref[u];
    const int b = s.fetch[((size_t)u * s.cap + e) * 2], slot = s.fetch[((size_t)u * s.cap + e) * 2 + 1];
    if (b < 0 || b >= nb_sel || slot < 0 || slot >= s.cslots) {
      if (tid == 0) atomicOr(s.err, kErrBounds);
      return j;
    }
    j.rows = b < geo.nb - 1 ? kBlock : (b == geo.nb - 1 ? geo.valid_tail : 0);
    j.src = reinterpret_cast<const uint4*>(s.host_kv + ((size_t)u * s.nb_max + b) * 2 * kBlockElems);
    j.dst = reinterpret_cast<uint4*>(s.cache + ((size_t)u * s.cslots + slot) * 2 * kBlockElems);
    return j;
  };
  auto load = [&](const Job& j, uint4 (&v)[kVec]) {
#pragma unroll
    for (int r = 0; r < kVec; ++r) {
      const int idx = tid + r * kGatherThreads;
      const int row = (idx >> 4) & (kBlock - 1);  // 16 vectors per 256-byte row; K rows then V rows
      v[r] = row < j.rows ? ld_stream_v4(j.src + idx) : make_uint4(0, 0, 0, 0);
    }
  };
  auto store = [&](const Job& j, const uint4 (&v)[kVec]) {
    if (j.rows < 0) return;
#pragma unroll
    for (int r = 0; r < kVec; ++r) j.dst[tid + r * kGatherThreads] = v[r];
  };
  uint4 va[kVec], vb[kVec];
  const int step = gridDim.x;
  Job ja = job(blockIdx.x);
  if (ja.rows >= 0) load(ja, va);
  for (int item = blockIdx.x; item < total; item += 2 * step) {
    const Job jb = job(item + step);  // the next item's loads go out before this item's stores
    if (jb.rows >= 0) load(jb, vb);
    store(ja, va);
    ja = job(item + 2 * step);
    if (ja.rows >= 0) load(ja, va);
    store(jb, vb);
  }
}

cudaError_t launch_gather(const LayerState& s, int ctas, cudaStream_t st, int ahead) {
  gather_kernel<<<ctas, kGatherThreads, 0, st>>>(s, ahead);
  return cudaGetLastError();
}

}  // namespace nosa
