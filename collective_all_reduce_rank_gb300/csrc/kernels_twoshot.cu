// kernels_twoshot.cu -- fused two-shot all-reduce.
//
// "Collective communication: NCCL's algorithms and protocols, and custom
// all-reduce in inference frameworks", section "Algorithms": in the first
// step each rank reads only 1/n of the other ranks' data and sums it (a
// reduce-scatter); in the second it reads the sums back (an all-gather);
// two synchronizations.
//
// One persistent cooperative launch of n x C CTAs.  CTA (r, ch) is channel
// ch of virtual rank r; its 16 warps are independent pipelines.  Each
// iteration a warp
//   1. reduces its part of tile t of chunk r over all n inputs (ascending
//      rank order) into outs[r], then releases its progress flag
//      (data -> release, the Simple protocol of the same page's
//      "Protocols" section);
//   2. for every other rank q, acquires the flag of warp w of CTA (q, ch)
//      for this iteration and copies that part of chunk q from outs[q] into
//      outs[r].
// Tile t of every chunk is handled by the same (channel, warp) in every
// rank, so the copy reads lines a sibling CTA wrote a moment earlier and
// finds them in L2.  No CTA-wide barrier is taken inside the loop.
#include "common.cuh"

namespace rra {

template <int N, int DT, bool VEC>
__device__ __forceinline__ void twoshot_warp(const TwoShotArgs& a, int r, int ch, int warp, int lane,
                                             int W, uint64_t E, uint32_t tag) {
  constexpr int PU = Elem<DT>::kPerUnit;
  constexpr int ES = Elem<DT>::kSize;
  constexpr int UPT = kTwoShotUnitsPerThread;
  const int C = a.channels;
  const size_t tile = (size_t)a.tile_units;
  const size_t wofs = (size_t)warp * 32 * UPT;
  const size_t per_iter = (size_t)C * tile;
  const size_t iters = ((a.chunk_len[0] + PU - 1) / PU + per_iter - 1) / per_iter;  // chunk 0 is the longest
  uint64_t* my_flag = a.progress + ((size_t)r * C + ch) * W + warp;
  const size_t lo = a.chunk_lo[r] * ES;
  const size_t len = a.chunk_len[r];
  // The inputs of iteration it+1 are loaded right after iteration it's
  // reduce, so their HBM latency overlaps the all-gather part of it.
  uint4 x[UPT][N];
  int v[UPT];
  auto load_x = [&](size_t it) {
    const size_t t0 = (it * C + ch) * tile + wofs;
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      const size_t u = t0 + (size_t)j * 32 + lane;
      v[j] = unit_valid<DT>(u, len);
      if (v[j] > 0) {
#pragma unroll
        for (int k = 0; k < N; ++k) x[j][k] = load_in<DT, VEC>(static_cast<const char*>(a.in[k]) + lo, u, v[j]);
      }
    }
  };
  if (iters > 0) load_x(0);

  for (size_t it = 0; it < iters; ++it) {
    const size_t t0 = (it * C + ch) * tile + wofs;
    // phase 1: reduce-scatter part
    {
#pragma unroll
      for (int j = 0; j < UPT; ++j) {
        if (v[j] > 0) {
          Acc s;
          acc_init<DT>(s, x[j][0]);
#pragma unroll
          for (int k = 1; k < N; ++k) acc_add<DT>(s, x[j][k]);
          const size_t u = t0 + (size_t)j * 32 + lane;
          store_out<DT, VEC, false>(static_cast<char*>(a.out[r]) + lo, u, v[j], acc_narrow<DT>(s));
        }
      }
    }
    __syncwarp();
    if (lane == 0) st_release(my_flag, E | (uint64_t)(it + 1));
    if (it + 1 < iters) load_x(it + 1);

    // phase 2: all-gather part.  Lane j waits for peer (r + j) mod N, so the
    // n-1 acquires run side by side; __syncwarp then orders every lane's
    // reads after all of them, and the n-1 tiles are read with all loads in
    // flight at once.
    {
      int ok = 1;
      if (lane >= 1 && lane < N) {
        const int q = (r + lane) % N;
        if (t0 < (a.chunk_len[q] + PU - 1) / PU) {
          uint64_t seen;
          ok = wait_geq(a.progress + ((size_t)q * C + ch) * W + warp, E | (uint64_t)(it + 1), &seen,
                        a.wait, tag, r, q, (int)it);
        }
      }
      ok = __all_sync(0xffffffffu, ok);
      __syncwarp();
      if (!ok) return;
    }
    uint4 y[N > 1 ? N - 1 : 1][UPT];
    int v[N > 1 ? N - 1 : 1][UPT];
#pragma unroll
    for (int j = 1; j < N; ++j) {
      const int q = (r + j) % N;
      const char* src = static_cast<const char*>(a.out[q]) + a.chunk_lo[q] * ES;
#pragma unroll
      for (int jj = 0; jj < UPT; ++jj) {
        const size_t u = t0 + (size_t)jj * 32 + lane;
        v[j - 1][jj] = unit_valid<DT>(u, a.chunk_len[q]);
        if (v[j - 1][jj] > 0) y[j - 1][jj] = load_shared_out<DT, VEC>(src, u, v[j - 1][jj]);
      }
    }
#pragma unroll
    for (int j = 1; j < N; ++j) {
      const int q = (r + j) % N;
      char* dst = static_cast<char*>(a.out[r]) + a.chunk_lo[q] * ES;
#pragma unroll
      for (int jj = 0; jj < UPT; ++jj) {
        const size_t u = t0 + (size_t)jj * 32 + lane;
        if (v[j - 1][jj] > 0) store_out<DT, VEC, true>(dst, u, v[j - 1][jj], y[j - 1][jj]);
      }
    }
  }
}

template <int N, int DT, bool VEC>
__global__ void __launch_bounds__(kDirectThreads, 1) twoshot_kernel(const __grid_constant__ TwoShotArgs a) {
  __shared__ uint32_t s_epoch;
  if (threadIdx.x == 0) s_epoch = read_epoch(a.wait.sync);
  __syncthreads();
  const uint32_t epoch = s_epoch;
  const int r = blockIdx.x % N, ch = blockIdx.x / N;
  const int W = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (r != a.wait.skip_rank)
    twoshot_warp<N, DT, VEC>(a, r, ch, warp, lane, W, (uint64_t)epoch << 32, epoch + 1u);
  arrive_end(a.wait.sync, epoch);
}

template <int N, int DT, bool VEC>
static const void* twoshot_fn() {
  return reinterpret_cast<const void*>(&twoshot_kernel<N, DT, VEC>);
}

template <int N>
static const void* twoshot_pick_n(int dt, bool vec) {
  if (dt == RRA_INT32) return vec ? twoshot_fn<N, RRA_INT32, true>() : twoshot_fn<N, RRA_INT32, false>();
  if (dt == RRA_FLOAT32) return vec ? twoshot_fn<N, RRA_FLOAT32, true>() : twoshot_fn<N, RRA_FLOAT32, false>();
  return vec ? twoshot_fn<N, RRA_BFLOAT16, true>() : twoshot_fn<N, RRA_BFLOAT16, false>();
}

static const void* twoshot_pick(int n, int dt, bool vec) {
  switch (n) {
    case 1: return twoshot_pick_n<1>(dt, vec);
    case 2: return twoshot_pick_n<2>(dt, vec);
    case 3: return twoshot_pick_n<3>(dt, vec);
    case 4: return twoshot_pick_n<4>(dt, vec);
    case 5: return twoshot_pick_n<5>(dt, vec);
    case 6: return twoshot_pick_n<6>(dt, vec);
    case 7: return twoshot_pick_n<7>(dt, vec);
    case 8: return twoshot_pick_n<8>(dt, vec);
    default: return nullptr;
  }
}

cudaError_t twoshot_occupancy(int n, int dt, bool vec, int* max_blocks_per_sm) {
  const void* f = twoshot_pick(n, dt, vec);
  if (!f) return cudaErrorInvalidValue;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(max_blocks_per_sm, f, kDirectThreads, 0);
}

cudaError_t launch_twoshot(int n, int dt, bool vec, const TwoShotArgs& a, int grid, cudaStream_t s) {
  const void* f = twoshot_pick(n, dt, vec);
  if (!f) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDirectThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<TwoShotArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, f, args);
}

}  // namespace rra
