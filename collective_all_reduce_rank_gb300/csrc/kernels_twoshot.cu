// kernels_twoshot.cu -- fused two-shot all-reduce.
//
// "Collective communication: NCCL's algorithms and protocols, and custom
// all-reduce in inference frameworks", section "Algorithms": in the first
// step each rank reads only 1/n of the other ranks' data and sums it (a
// reduce-scatter); in the second it reads the sums back (an all-gather);
// two synchronizations.
//
// One persistent cooperative launch of n x C CTAs, two per SM.  CTA (r, ch)
// is channel ch of virtual rank r.  Up to four ranks (the fused form) its
// 16 warps are independent pipelines, each lane with 2 (two ranks) or 1
// 16-byte units per tile; from five ranks (the split form, below) 8 warps
// reduce and 8 gather.  In the fused form warp w handles its part of tile t of
// every chunk in turn and, in trip i of its loop,
//   1. issues the loads of the all-gather part of tile i - F: the other
//      ranks' sums, from outs[q] (L2), after acquiring their progress;
//   2. reduces tile i of chunk r over all n inputs (ascending rank order,
//      inputs loaded one trip ahead) into outs[r];
//   3. issues the input loads of tile i + 1;
//   4. stores the gathered sums of tile i - F into outs[r];
//   5. every F tiles, fences and raises its progress flag to the tiles
//      reduced so far (data -> release, the Simple protocol of the same
//      page's "Protocols" section).
// The gather trails the reduce by F tiles, so the flags it needs were
// posted F tiles earlier and it rarely waits; one fence covers F tiles; the
// L2 loads of the gather and the HBM loads of the next inputs are in flight
// together.  Tile t of every chunk is handled by the same (channel, warp)
// in every rank, so the gather reads lines a sibling CTA wrote a moment
// earlier and finds them in L2.  No CTA-wide barrier is taken in the loop.
#include "common.cuh"

namespace rra {

// F: tiles between progress flags and of gather lag (measured on GB300: 16
// for eight ranks, 8 for fewer)
template <int N>
__host__ __device__ constexpr int twoshot_lag() {
  return N >= 8 ? 16 : 8;
}

template <int N, int DT, bool VEC>
__device__ __forceinline__ void twoshot_warp(const TwoShotArgs& a, int r, int ch, int warp, int lane,
                                             int W, uint64_t E, uint32_t tag) {
  constexpr int PU = Elem<DT>::kPerUnit;
  constexpr int ES = Elem<DT>::kSize;
  // the measured default, or the host's (RRA_TWOSHOT_LAG)
  const size_t F = a.lag > 0 ? (size_t)a.lag : (size_t)twoshot_lag<N>();
  constexpr int UPT = twoshot_units_per_thread(N);  // units per lane per tile
  constexpr int NY = N > 1 ? N - 1 : 1;
  const int C = a.channels;
  const size_t tile = (size_t)a.tile_units;  // = threads * UPT
  const size_t per_iter = (size_t)C * tile;
  const size_t iters = ((a.chunk_len[0] + PU - 1) / PU + per_iter - 1) / per_iter;  // chunk 0 is the longest
  uint64_t* my_flag = a.progress + ((size_t)r * C + ch) * W + warp;
  const size_t lo = a.chunk_lo[r] * ES;
  const size_t len = a.chunk_len[r];
  // first unit of this warp's part of tile `it`; lane unit j is + 32j + lane
  auto first_of = [&](size_t it) { return (it * C + ch) * tile + (size_t)warp * 32 * UPT; };

  uint4 x[UPT][N];
  int v[UPT];
  auto load_x = [&](size_t it) {
    const size_t u0 = first_of(it) + lane;
#pragma unroll
    for (int j = 0; j < UPT; ++j) {
      const size_t u = u0 + 32 * j;
      v[j] = unit_valid<DT>(u, len);
      if (v[j] > 0) {
#pragma unroll
        for (int k = 0; k < N; ++k) x[j][k] = load_in<DT, VEC>(static_cast<const char*>(a.in[k]) + lo, u, v[j]);
      }
    }
  };
  if (iters > 0) load_x(0);
  uint64_t seen = 0;  // polling lane j's last observed value of peer (r + j)'s flag
  size_t due = F;     // reduced tiles after which the next progress flag goes up

  for (size_t it = 0; it < iters + F; ++it) {
    // 1. gather loads of tile gi = it - F
    const bool gather = it >= F;
    const size_t gi = it - F;
    uint4 y[UPT][NY];
    int vy[UPT][NY];
    if (gather) {
      int ok = 1;
      if (lane >= 1 && lane < N) {
        const int q = (r + lane) % N;
        const uint64_t want = E | (uint64_t)(gi + 1);
        if (first_of(gi) < (a.chunk_len[q] + PU - 1) / PU && seen < want)
          ok = wait_geq(a.progress + ((size_t)q * C + ch) * W + warp, want, &seen, a.wait, tag, r, q, (int)gi);
      }
      ok = __all_sync(0xffffffffu, ok);
      __syncwarp();
      if (!ok) return;
      const size_t u0 = first_of(gi) + lane;
#pragma unroll
      for (int i = 1; i < N; ++i) {
        const int q = (r + i) % N;
        const char* src = static_cast<const char*>(a.out[q]) + a.chunk_lo[q] * ES;
#pragma unroll
        for (int j = 0; j < UPT; ++j) {
          vy[j][i - 1] = unit_valid<DT>(u0 + 32 * j, a.chunk_len[q]);
          if (vy[j][i - 1] > 0) y[j][i - 1] = load_shared_out<DT, VEC>(src, u0 + 32 * j, vy[j][i - 1]);
        }
      }
    }
    // 2-3. reduce tile it, then load the inputs of tile it + 1
    const bool reduce = it < iters;
    if (reduce) {
      const size_t u0 = first_of(it) + lane;
#pragma unroll
      for (int j = 0; j < UPT; ++j) {
        if (v[j] > 0) {
          Acc s;
          acc_init<DT>(s, x[j][0]);
#pragma unroll
          for (int k = 1; k < N; ++k) acc_add<DT>(s, x[j][k]);
          store_out<DT, VEC, false>(static_cast<char*>(a.out[r]) + lo, u0 + 32 * j, v[j], acc_narrow<DT>(s));
        }
      }
      if (it + 1 < iters) load_x(it + 1);
    }
    // 4. gathered sums into this rank's output
    if (gather) {
      const size_t u0 = first_of(gi) + lane;
#pragma unroll
      for (int i = 1; i < N; ++i) {
        const int q = (r + i) % N;
        char* dst = static_cast<char*>(a.out[r]) + a.chunk_lo[q] * ES;
#pragma unroll
        for (int j = 0; j < UPT; ++j)
          if (vy[j][i - 1] > 0) store_out<DT, VEC, true>(dst, u0 + 32 * j, vy[j][i - 1], y[j][i - 1]);
      }
    }
    // 5. progress: tiles 0..it reduced (every F tiles and after the last)
    if (reduce && (it + 1 == due || it + 1 == iters)) {
      __syncwarp();
      if (lane == 0) st_release(my_flag, E | (uint64_t)(it + 1));
      due += F;
    }
    // trips after the last reduce and before the first gather do nothing
    if (it + 1 >= iters && it + 1 < F) it = F - 1;
  }
}

// Split form (five ranks and more): warps 0..W/2-1 reduce, warp W/2 + w
// gathers what reducer w of every other rank posts.  Reducers never wait;
// a gatherer waits on the peers' progress flags of its pipeline.
template <int N, int DT, bool VEC>
__device__ __forceinline__ void twoshot_split_warp(const TwoShotArgs& a, int r, int ch, int warp, int lane,
                                                   int W, uint64_t E, uint32_t tag) {
  constexpr int PU = Elem<DT>::kPerUnit;
  constexpr int ES = Elem<DT>::kSize;
  const size_t F = a.lag > 0 ? (size_t)a.lag : (size_t)twoshot_lag<N>();
  const int WR = W / 2;
  const bool reducer = warp < WR;
  const int pw = reducer ? warp : warp - WR;  // pipeline
  const int C = a.channels;
  const size_t tile = (size_t)a.tile_units;  // = WR * 32
  const size_t per_iter = (size_t)C * tile;
  const size_t iters = ((a.chunk_len[0] + PU - 1) / PU + per_iter - 1) / per_iter;  // chunk 0 is the longest
  auto first_of = [&](size_t it) { return (it * C + ch) * tile + (size_t)pw * 32; };
  if (reducer) {
    uint64_t* my_flag = a.progress + ((size_t)r * C + ch) * W + pw;
    const size_t lo = a.chunk_lo[r] * ES;
    const size_t len = a.chunk_len[r];
    uint4 x[N];
    int v = 0;
    auto load_x = [&](size_t it) {
      const size_t u = first_of(it) + lane;
      v = unit_valid<DT>(u, len);
      if (v > 0) {
#pragma unroll
        for (int k = 0; k < N; ++k) x[k] = load_in<DT, VEC>(static_cast<const char*>(a.in[k]) + lo, u, v);
      }
    };
    if (iters > 0) load_x(0);
    size_t due = F;
    for (size_t it = 0; it < iters; ++it) {
      if (v > 0) {
        Acc s;
        acc_init<DT>(s, x[0]);
#pragma unroll
        for (int k = 1; k < N; ++k) acc_add<DT>(s, x[k]);
        store_out<DT, VEC, false>(static_cast<char*>(a.out[r]) + lo, first_of(it) + lane, v, acc_narrow<DT>(s));
      }
      if (it + 1 < iters) load_x(it + 1);
      if (it + 1 == due || it + 1 == iters) {
        __syncwarp();
        if (lane == 0) st_release(my_flag, E | (uint64_t)(it + 1));
        due += F;
      }
    }
    return;
  }
  uint64_t seen = 0;  // polling lane j's last observed value of peer (r + j)'s flag
  for (size_t gi = 0; gi < iters; ++gi) {
    int ok = 1;
    if (lane >= 1 && lane < N) {
      const int q = (r + lane) % N;
      const uint64_t want = E | (uint64_t)(gi + 1);
      if (first_of(gi) < (a.chunk_len[q] + PU - 1) / PU && seen < want)
        ok = wait_geq(a.progress + ((size_t)q * C + ch) * W + pw, want, &seen, a.wait, tag, r, q, (int)gi);
    }
    ok = __all_sync(0xffffffffu, ok);
    __syncwarp();
    if (!ok) return;
    const size_t u = first_of(gi) + lane;
    uint4 y[N - 1];
    int vy[N - 1];
#pragma unroll
    for (int i = 1; i < N; ++i) {
      const int q = (r + i) % N;
      const char* src = static_cast<const char*>(a.out[q]) + a.chunk_lo[q] * ES;
      vy[i - 1] = unit_valid<DT>(u, a.chunk_len[q]);
      if (vy[i - 1] > 0) y[i - 1] = load_shared_out<DT, VEC>(src, u, vy[i - 1]);
    }
#pragma unroll
    for (int i = 1; i < N; ++i) {
      const int q = (r + i) % N;
      char* dst = static_cast<char*>(a.out[r]) + a.chunk_lo[q] * ES;
      if (vy[i - 1] > 0) store_out<DT, VEC, true>(dst, u, vy[i - 1], y[i - 1]);
    }
  }
}

template <int N, int DT, bool VEC>
__global__ void __launch_bounds__(kDirectThreads, twoshot_min_blocks(N)) twoshot_kernel(const __grid_constant__ TwoShotArgs a) {
  __shared__ uint32_t s_epoch;
  if (threadIdx.x == 0) s_epoch = read_epoch(a.wait.sync);
  __syncthreads();
  const uint32_t epoch = s_epoch;
  const int r = blockIdx.x % N, ch = blockIdx.x / N;
  const int W = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (r != a.wait.skip_rank) {
    if constexpr (twoshot_split(N))
      twoshot_split_warp<N, DT, VEC>(a, r, ch, warp, lane, W, (uint64_t)epoch << 32, epoch + 1u);
    else
      twoshot_warp<N, DT, VEC>(a, r, ch, warp, lane, W, (uint64_t)epoch << 32, epoch + 1u);
  }
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
