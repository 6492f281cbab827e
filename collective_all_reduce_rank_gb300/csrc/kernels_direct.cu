// kernels_direct.cu -- one-shot all-reduce, direct reduce-scatter, direct
// all-gather.
//
// One-shot ("Collective communication: NCCL's algorithms and protocols...",
// section "Algorithms"): every rank reads the full data of the other n-1
// ranks and sums locally.  All n virtual ranks share one HBM here, so rank
// r's n reads of a tile are the same bytes as rank q's: a thread reads each
// of the n inputs of its 16-byte unit once, sums them in ascending rank
// order (the order every rank uses), and stores the one sum to all n
// outputs.  That is the one-shot result bit for bit at the HBM floor of
// n reads + n writes per unit.  per_rank_grid = 1 launches the literal
// form instead: grid row r computes rank r's output only (n^2 reads, which
// the L2 mostly absorbs).
//
// Direct reduce-scatter and all-gather are the two halves of two-shot
// (same page, "Algorithms": reduce your 1/n slice, then read the sums
// back), exposed on their own.
#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "common.cuh"

namespace rra {

// Up to four ranks (three for bfloat16) a thread takes two units per trip
// (2n loads in flight); above, the kernel is built for two CTAs per SM with
// one unit per trip (n loads a thread, 53-60 registers at eight ranks
// against 94): on GB300 at 8 ranks x 8 MiB fp32 0.85 -> 0.90 of the HBM
// copy rate, bf16 at 64-256 MiB 0.88-0.92 -> 0.90-0.93, fp32 at 64-256 MiB
// within 0.5%.  bfloat16 at four ranks (78 registers with two units, one
// CTA per SM; 44 with one): 16 MiB-1 GiB 0.89-0.99 -> 0.95-1.05; at two
// and three ranks one unit measured 3-13% slower.
template <int N, int DT>
__host__ __device__ constexpr bool oneshot_two_units() {
  return DT == RRA_BFLOAT16 ? N <= 3 : N <= 4;
}

template <int N, int DT, bool VEC>
__global__ void __launch_bounds__(kDirectThreads, oneshot_two_units<N, DT>() ? 1 : 2)
    oneshot_kernel(const __grid_constant__ DirectArgs a) {
  const size_t count = a.count;
  const size_t units = (count + Elem<DT>::kPerUnit - 1) / Elem<DT>::kPerUnit;
  int r_lo = 0, r_hi = N;
  if (a.per_rank_grid) {
    r_lo = blockIdx.y;
    r_hi = r_lo + 1;
  }
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t u = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  // two units per trip: 2N independent 16-byte loads in flight per thread
  for (; oneshot_two_units<N, DT>() && u + stride < units; u += 2 * stride) {
    const size_t u1 = u + stride;
    const int v0 = unit_valid<DT>(u, count), v1 = unit_valid<DT>(u1, count);
    uint4 x0[N], x1[N];
#pragma unroll
    for (int k = 0; k < N; ++k) {
      x0[k] = load_in<DT, VEC>(a.in[k], u, v0);
      x1[k] = load_in<DT, VEC>(a.in[k], u1, v1);
    }
    Acc s0, s1;
    acc_init<DT>(s0, x0[0]);
    acc_init<DT>(s1, x1[0]);
#pragma unroll
    for (int k = 1; k < N; ++k) {
      acc_add<DT>(s0, x0[k]);
      acc_add<DT>(s1, x1[k]);
    }
    const uint4 y0 = acc_narrow<DT>(s0), y1 = acc_narrow<DT>(s1);
    for (int r = r_lo; r < r_hi; ++r) {
      store_out<DT, VEC, true>(a.out[r], u, v0, y0);
      store_out<DT, VEC, true>(a.out[r], u1, v1, y1);
    }
  }
  for (; u < units; u += stride) {
    const int v0 = unit_valid<DT>(u, count);
    uint4 x0[N];
#pragma unroll
    for (int k = 0; k < N; ++k) x0[k] = load_in<DT, VEC>(a.in[k], u, v0);
    Acc s0;
    acc_init<DT>(s0, x0[0]);
#pragma unroll
    for (int k = 1; k < N; ++k) acc_add<DT>(s0, x0[k]);
    const uint4 y0 = acc_narrow<DT>(s0);
    for (int r = r_lo; r < r_hi; ++r) store_out<DT, VEC, true>(a.out[r], u, v0, y0);
  }
}

// Direct reduce-scatter: grid row r = blockIdx.y computes
// out[r][i] = SUM_k in[k][r*rc + i] in ascending rank order.
template <int N, int DT, bool VEC>
__global__ void __launch_bounds__(kDirectThreads) direct_rs_kernel(const __grid_constant__ DirectArgs a) {
  const size_t rc = a.count;
  const size_t units = (rc + Elem<DT>::kPerUnit - 1) / Elem<DT>::kPerUnit;
  const int r = blockIdx.y;
  const size_t slice_off = (size_t)r * rc * Elem<DT>::kSize;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t u = (size_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += stride) {
    const int v = unit_valid<DT>(u, rc);
    uint4 x[N];
#pragma unroll
    for (int k = 0; k < N; ++k)
      x[k] = load_in<DT, VEC>(static_cast<const char*>(a.in[k]) + slice_off, u, v);
    Acc s;
    acc_init<DT>(s, x[0]);
#pragma unroll
    for (int k = 1; k < N; ++k) acc_add<DT>(s, x[k]);
    store_out<DT, VEC, true>(a.out[r], u, v, acc_narrow<DT>(s));
  }
}

// Direct all-gather: grid row q = blockIdx.y reads shard q once and stores
// it into every rank's output at q*sc.
template <int N, int DT, bool VEC>
__global__ void __launch_bounds__(kDirectThreads) direct_ag_kernel(const __grid_constant__ DirectArgs a) {
  const size_t sc = a.count;
  const size_t units = (sc + Elem<DT>::kPerUnit - 1) / Elem<DT>::kPerUnit;
  const int q = blockIdx.y;
  const size_t dst_off = (size_t)q * sc * Elem<DT>::kSize;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t u = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; u + stride < units; u += 2 * stride) {
    const size_t u1 = u + stride;
    const int v0 = unit_valid<DT>(u, sc), v1 = unit_valid<DT>(u1, sc);
    const uint4 x0 = load_in<DT, VEC>(a.in[q], u, v0);
    const uint4 x1 = load_in<DT, VEC>(a.in[q], u1, v1);
#pragma unroll
    for (int r = 0; r < N; ++r) {
      store_out<DT, VEC, true>(static_cast<char*>(a.out[r]) + dst_off, u, v0, x0);
      store_out<DT, VEC, true>(static_cast<char*>(a.out[r]) + dst_off, u1, v1, x1);
    }
  }
  if (u < units) {
    const int v0 = unit_valid<DT>(u, sc);
    const uint4 x0 = load_in<DT, VEC>(a.in[q], u, v0);
#pragma unroll
    for (int r = 0; r < N; ++r) store_out<DT, VEC, true>(static_cast<char*>(a.out[r]) + dst_off, u, v0, x0);
  }
}

// ---------------------------------------------------------------------------
// dispatch.  Grid: for calls that move at least `cover_from` floor bytes, a
// covering grid (every thread one trip of `upt` units), so the block
// scheduler hands tiles out as SMs free up; a resident grid (occupancy of
// the exact instance x SM count / rows, grid-stride) splits them statically
// and waits for its slowest CTAs.  Measured on GB300, covering against
// resident, fraction of the HBM copy rate from 64 MiB to 1 GiB per rank at
// 2-8 ranks: one-shot 0.82-0.96 -> 0.89-1.05, direct reduce-scatter
// 0.94-0.99 -> 0.98-1.05, direct all-gather 0.77-0.90 -> 0.86-1.03.  Below
// the thresholds (256 MB of floor bytes for one-shot, 64 MB for the
// reduce-scatter and all-gather) the resident grid measured as fast or up
// to 13% faster.  An SM budget (rra_set_max_ctas) keeps the resident grid;
// RRA_DIRECT_GRID=resident | cover forces one form at every size.
// ---------------------------------------------------------------------------
static int device_sms() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

template <typename Kern>
static int occupancy_of(Kern k) {
  int b = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k, kDirectThreads, 0) != cudaSuccess || b < 1) b = 1;
  return b;
}

// RRA_DIRECT_GRID, read at every call: 0 by size, 1 resident, 2 cover
static int forced_grid() {
  const char* e = std::getenv("RRA_DIRECT_GRID");
  if (!e) return 0;
  if (!std::strcmp(e, "resident")) return 1;
  if (!std::strcmp(e, "cover")) return 2;
  return 0;
}

static int grid_for(size_t units, int occ, int rows, int upt, size_t floor_bytes, size_t cover_from) {
  const size_t want = (units + kDirectThreads - 1) / kDirectThreads;
  int per_row = std::max(1, device_sms() * occ / rows);
  const int forced = forced_grid();
  if (max_ctas_cap() > 0) {
    per_row = std::max(1, std::min(per_row, max_ctas_cap() / rows));
  } else if (forced == 2 || (forced == 0 && floor_bytes >= cover_from)) {
    const size_t cover = (units + (size_t)kDirectThreads * upt - 1) / ((size_t)kDirectThreads * upt);
    return (int)std::max<size_t>(1, std::min<size_t>(cover, 0x7fffffff));
  }
  return (int)std::max<size_t>(1, std::min(want, (size_t)per_row));
}

#define RRA_DIRECT_DISPATCH(KERNEL, UPT, FLOOR_PER_UNIT, COVER_FROM)                      \
  template <int N, int DT, bool VEC>                                                         \
  static cudaError_t KERNEL##_go(const DirectArgs& a, size_t units, int rows, int* grid,     \
                                 cudaStream_t s) {                                           \
    static const int occ = occupancy_of(KERNEL<N, DT, VEC>);                                 \
    *grid = grid_for(units, occ, rows, UPT, units * (FLOOR_PER_UNIT), COVER_FROM);           \
    KERNEL<N, DT, VEC><<<dim3(*grid, rows), kDirectThreads, 0, s>>>(a);                      \
    return cudaGetLastError();                                                               \
  }                                                                                          \
  template <int N>                                                                           \
  static cudaError_t KERNEL##_launch_n(int dt, bool vec, const DirectArgs& a, size_t units,  \
                                       int rows, int* grid, cudaStream_t s) {                \
    if (dt == RRA_INT32)                                                                     \
      return vec ? KERNEL##_go<N, RRA_INT32, true>(a, units, rows, grid, s)                  \
                 : KERNEL##_go<N, RRA_INT32, false>(a, units, rows, grid, s);                \
    if (dt == RRA_FLOAT32)                                                                   \
      return vec ? KERNEL##_go<N, RRA_FLOAT32, true>(a, units, rows, grid, s)                \
                 : KERNEL##_go<N, RRA_FLOAT32, false>(a, units, rows, grid, s);              \
    return vec ? KERNEL##_go<N, RRA_BFLOAT16, true>(a, units, rows, grid, s)                 \
               : KERNEL##_go<N, RRA_BFLOAT16, false>(a, units, rows, grid, s);               \
  }                                                                                          \
  static cudaError_t KERNEL##_launch(int n, int dt, bool vec, const DirectArgs& a,           \
                                     size_t units, int rows, int* grid, cudaStream_t s) {    \
    switch (n) {                                                                             \
      case 1: return KERNEL##_launch_n<1>(dt, vec, a, units, rows, grid, s);                 \
      case 2: return KERNEL##_launch_n<2>(dt, vec, a, units, rows, grid, s);                 \
      case 3: return KERNEL##_launch_n<3>(dt, vec, a, units, rows, grid, s);                 \
      case 4: return KERNEL##_launch_n<4>(dt, vec, a, units, rows, grid, s);                 \
      case 5: return KERNEL##_launch_n<5>(dt, vec, a, units, rows, grid, s);                 \
      case 6: return KERNEL##_launch_n<6>(dt, vec, a, units, rows, grid, s);                 \
      case 7: return KERNEL##_launch_n<7>(dt, vec, a, units, rows, grid, s);                 \
      case 8: return KERNEL##_launch_n<8>(dt, vec, a, units, rows, grid, s);                 \
      default: return cudaErrorInvalidValue;                                                 \
    }                                                                                        \
  }

// Per kernel: units a thread takes in one trip (one-shot two up to four
// ranks, three for bfloat16; the reduce-scatter one, the all-gather two);
// floor bytes per unit
// of `units` (one-shot: n reads and n writes of each unit; reduce-scatter
// and all-gather, `units` being one rank's slice: (n + 1) n bytes of each);
// the floor bytes from which the grid covers.
RRA_DIRECT_DISPATCH(oneshot_kernel, (oneshot_two_units<N, DT>() ? 2 : 1), 2 * N * 16, (size_t)256 << 20)
RRA_DIRECT_DISPATCH(direct_rs_kernel, 1, (N + 1) * N * 16, (size_t)64 << 20)
RRA_DIRECT_DISPATCH(direct_ag_kernel, 2, (N + 1) * N * 16, (size_t)64 << 20)

cudaError_t launch_oneshot(int n, int dt, bool vec, const DirectArgs& a, size_t units, int* grid,
                           cudaStream_t s) {
  return oneshot_kernel_launch(n, dt, vec, a, units, a.per_rank_grid ? n : 1, grid, s);
}

cudaError_t launch_direct_rs(int n, int dt, bool vec, const DirectArgs& a, size_t units, int* grid,
                             cudaStream_t s) {
  return direct_rs_kernel_launch(n, dt, vec, a, units, n, grid, s);
}

cudaError_t launch_direct_ag(int n, int dt, bool vec, const DirectArgs& a, size_t units, int* grid,
                             cudaStream_t s) {
  return direct_ag_kernel_launch(n, dt, vec, a, units, n, grid, s);
}

}  // namespace rra
