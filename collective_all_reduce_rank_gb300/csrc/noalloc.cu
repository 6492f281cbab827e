// noalloc.cu -- an all-reduce entry point that allocates nothing.
//
// rra_allreduce_two_shot_static runs the two-shot kernel with its scratch
// (status block, call epoch, per-(rank, channel, warp) progress flags) in a
// file-scope __device__ array instead of the workspace rra_init allocates.
// It serves callers that may not allocate device memory themselves.
//
// The array lives in the module's static device memory: every GPU that
// loads librra.so holds kStaticScratchBytes of it until the process exits.
// In host code `g_static_scratch` names a host-side stand-in, not the
// device array, so host code never passes it to a kernel: the device
// address comes from cudaGetSymbolAddress, taken once per device.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "rra.h"
#include "rra_internal.h"

namespace rra {
namespace {

constexpr int kStaticMaxChannels = 16;
constexpr size_t kStaticFlagWords = (size_t)kMaxRanks * kStaticMaxChannels * kMaxWarps;  // 2048
constexpr size_t kStaticFlagOffset = 256;
constexpr size_t kStaticScratchBytes = kStaticFlagOffset + kStaticFlagWords * sizeof(uint64_t);  // 16640
constexpr uint64_t kStaticTimeoutNs = 500ull * 1000 * 1000;
constexpr int kMaxDevices = 64;

// [0, 64): DevStatus   [64, 128): SyncHdr   [256, ...): progress flags
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_setup_mu;
std::atomic<char*> g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device, looked up
// once per device (with that device current).
cudaError_t scratch_for_current_device(char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  char* p = g_scratch_ptr[dev].load();
  if (!p) {
    std::lock_guard<std::mutex> lk(g_setup_mu);
    p = g_scratch_ptr[dev].load();
    if (!p) {
      void* addr = nullptr;
      e = cudaGetSymbolAddress(&addr, g_static_scratch);
      if (e != cudaSuccess) return e;
      if (!addr) return cudaErrorInvalidSymbol;
      p = static_cast<char*>(addr);
      g_scratch_ptr[dev].store(p);
    }
  }
  *out = p;
  return cudaSuccess;
}

bool ranges_overlap(const void* a, size_t an, const void* b, size_t bn) {
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return an && bn && x < y + bn && y < x + an;
}

}  // namespace
}  // namespace rra

using namespace rra;

extern "C" rra_status_t rra_allreduce_two_shot_static(const void* const* bufs, void* const* outs,
                                                      int nranks, size_t count, rra_dtype_t dtype,
                                                      rra_op_t op, rra_stream_t stream) {
  if (!bufs || !outs || nranks < 1 || op != RRA_SUM ||
      (dtype != RRA_INT32 && dtype != RRA_FLOAT32 && dtype != RRA_BFLOAT16))
    return RRA_ERR_INVALID_ARG;
  if (nranks > kMaxRanks) return RRA_ERR_UNSUPPORTED;  // the static flags hold 8 ranks at most
  const size_t e = dtype == RRA_BFLOAT16 ? 2 : 4;
  if (count > (SIZE_MAX / 2) / e) return RRA_ERR_INVALID_ARG;
  const size_t S = count * e;
  for (int r = 0; r < nranks; ++r)
    if (!bufs[r] || !outs[r] || (uintptr_t)bufs[r] % e || (uintptr_t)outs[r] % e) return RRA_ERR_INVALID_ARG;
  for (int i = 0; i < nranks; ++i)
    for (int j = 0; j < nranks; ++j) {
      if (i < j && ranges_overlap(outs[i], S, outs[j], S)) return RRA_ERR_ALIAS;
      if (ranges_overlap(outs[j], S, bufs[i], S) && !(i == j && outs[j] == bufs[i])) return RRA_ERR_ALIAS;
    }
  if (count == 0) return RRA_SUCCESS;

  char* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return RRA_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  TwoShotArgs a{};
  const size_t pu = 16 / e;
  const size_t per = (count + nranks - 1) / nranks;
  const size_t clen = (per + pu - 1) / pu * pu;
  bool vec = true;
  for (int c = 0; c < nranks; ++c) {
    a.in[c] = bufs[c];
    a.out[c] = outs[c];
    const size_t lo = c * clen < count ? c * clen : count;
    const size_t hi = (c + 1) * clen < count ? (c + 1) * clen : count;
    a.chunk_lo[c] = lo;
    a.chunk_len[c] = hi - lo;
    vec = vec && (uintptr_t)bufs[c] % 16 == 0 && (uintptr_t)outs[c] % 16 == 0;
  }
  a.tile_units = kDirectThreads * twoshot_units_per_thread(nranks);
  int occ = 0, dev = 0, sms = 0;
  if (twoshot_occupancy(nranks, dtype, vec, &occ) != cudaSuccess || occ < 1) return RRA_ERR_CUDA;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t units0 = (a.chunk_len[0] + pu - 1) / pu;
  size_t c = (units0 + a.tile_units - 1) / a.tile_units;
  if (c < 1) c = 1;
  if (c > (size_t)kStaticMaxChannels) c = kStaticMaxChannels;
  if (c > (size_t)(sms * occ / nranks)) c = (size_t)(sms * occ / nranks);
  if (c < 1) return RRA_ERR_UNSUPPORTED;
  if ((size_t)nranks * c * kMaxWarps > kStaticFlagWords) return RRA_ERR_UNSUPPORTED;
  a.channels = (int)c;
  a.progress = reinterpret_cast<uint64_t*>(scratch + kStaticFlagOffset);
  a.wait.status = reinterpret_cast<DevStatus*>(scratch);
  a.wait.sync = reinterpret_cast<SyncHdr*>(scratch + 64);
  a.wait.timeout_ns = kStaticTimeoutNs;
  a.wait.skip_rank = -1;
  // The status block must start each call at zero; the epoch and the
  // arrival counter carry over (the last CTA of each call resets the
  // counter and bumps the epoch, so the flags never need clearing).
  if (cudaMemsetAsync(scratch, 0, sizeof(DevStatus), st) != cudaSuccess) return RRA_ERR_CUDA;
  if (launch_twoshot(nranks, dtype, vec, a, nranks * (int)c, st) != cudaSuccess) return RRA_ERR_CUDA;
  return RRA_SUCCESS;
}
