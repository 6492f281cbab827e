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

cudaStream_t stream_of(rra_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

constexpr const char* kCall = "allreduce_two_shot_static";

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
  auto fail = [&](rra_status_t e) { return record_call(kCall, RRA_ALGO_TWO_SHOT, nranks, count, dtype, 0, e); };
  if (!bufs || !outs || nranks < 1 || op != RRA_SUM ||
      (dtype != RRA_INT32 && dtype != RRA_FLOAT32 && dtype != RRA_BFLOAT16))
    return fail(nranks > kMaxRanks ? RRA_ERR_UNSUPPORTED : RRA_ERR_INVALID_ARG);
  if (nranks > kMaxRanks) return fail(RRA_ERR_UNSUPPORTED);  // the static flags hold 8 ranks at most
  const size_t e = dtype == RRA_BFLOAT16 ? 2 : 4;
  if (count > (SIZE_MAX / 2) / e) return fail(RRA_ERR_INVALID_ARG);
  const size_t S = count * e;
  for (int r = 0; r < nranks; ++r)
    if (!bufs[r] || !outs[r] || (uintptr_t)bufs[r] % e || (uintptr_t)outs[r] % e) return fail(RRA_ERR_INVALID_ARG);
  for (int i = 0; i < nranks; ++i)
    for (int j = 0; j < nranks; ++j) {
      if (i < j && ranges_overlap(outs[i], S, outs[j], S)) return fail(RRA_ERR_ALIAS);
      if (ranges_overlap(outs[j], S, bufs[i], S) && !(i == j && outs[j] == bufs[i])) return fail(RRA_ERR_ALIAS);
    }
  if (count == 0) return fail(RRA_SUCCESS);

  char* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess)
    return record_call(kCall, RRA_ALGO_TWO_SHOT, nranks, count, dtype, 0, RRA_ERR_CUDA);

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
  a.tile_units = twoshot_tile_units(nranks);
  int occ = 0, dev = 0, sms = 0;
  if (twoshot_occupancy(nranks, dtype, vec, &occ) != cudaSuccess || occ < 1)
    return record_call(kCall, RRA_ALGO_TWO_SHOT, nranks, count, dtype, 0, RRA_ERR_CUDA);
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t units0 = (a.chunk_len[0] + pu - 1) / pu;
  size_t c = (units0 + a.tile_units - 1) / a.tile_units;
  if (c < 1) c = 1;
  if (c > (size_t)kStaticMaxChannels) c = kStaticMaxChannels;
  if (c > (size_t)(sms * occ / nranks)) c = (size_t)(sms * occ / nranks);
  if (c > (size_t)channels_allowed(nranks)) c = (size_t)channels_allowed(nranks);  // the SM budget
  if (c < 1 || (size_t)nranks * c * kMaxWarps > kStaticFlagWords)
    return record_call(kCall, RRA_ALGO_TWO_SHOT, nranks, count, dtype, 0, RRA_ERR_UNSUPPORTED);
  a.channels = (int)c;
  a.progress = reinterpret_cast<uint64_t*>(scratch + kStaticFlagOffset);
  a.wait.status = reinterpret_cast<DevStatus*>(scratch);
  a.wait.sync = reinterpret_cast<SyncHdr*>(scratch + 64);
  a.wait.timeout_ns = current_timeout_ns();
  a.wait.skip_rank = current_skip_rank();
  // The status block keeps the first device error until
  // rra_query_status_static reads and clears it (a stale abort tag never
  // matches a later call's tag); the epoch and the arrival counter carry
  // over (the last CTA of each call resets the counter and bumps the epoch,
  // so the flags never need clearing).
  const rra_status_t st = launch_twoshot(nranks, dtype, vec, a, nranks * (int)c, stream_of(stream)) == cudaSuccess
                              ? RRA_SUCCESS
                              : RRA_ERR_CUDA;
  return record_call(kCall, RRA_ALGO_TWO_SHOT, nranks, count, dtype, nranks * (int)c, st);
}

extern "C" rra_status_t rra_query_status_static(rra_stream_t stream, int32_t info[4]) {
  if (info) info[0] = info[1] = info[2] = info[3] = 0;
  if (cudaStreamSynchronize(stream_of(stream)) != cudaSuccess) return RRA_ERR_CUDA;
  char* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return RRA_ERR_CUDA;
  DevStatus h{};
  if (cudaMemcpy(&h, scratch, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return RRA_ERR_CUDA;
  if (h.code == 0) return RRA_SUCCESS;
  if (info) decode_status(h, info);
  // clear the record; the abort tag belongs to a finished call and can stay
  DevStatus z{};
  z.abort_tag = h.abort_tag;
  if (cudaMemcpy(scratch, &z, sizeof z, cudaMemcpyHostToDevice) != cudaSuccess) return RRA_ERR_CUDA;
  return (rra_status_t)h.code;
}
