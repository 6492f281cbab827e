// kernels_rmsnorm.cu -- all-reduce fused with RMSNorm over rows.
//
// "Collective communication: NCCL's algorithms and protocols, and custom
// all-reduce in inference frameworks", section "Source code": FlashInfer's
// fused all-reduce + RMSNorm, used on tensor-parallel activations
// [tokens, hidden] right after the row-parallel layer's all-reduce.
//
// One CTA per row.  Pass 1 sums the row of the n inputs (one-shot: each
// 16-byte unit of every input read once, float32, ascending rank order),
// keeps the float32 sums in shared memory and accumulates their squares.
// After a block reduction, pass 2 scales every sum by
// rsqrt(mean square + eps) and gamma and stores the rounded row to all n
// outputs.  Saves the separate normalisation kernel's full re-read and
// re-write of the activations.
#include "common.cuh"

namespace rra {

constexpr int kNormThreads = 256;

struct NormArgs {
  const void* in[kMaxRanks];
  void* out[kMaxRanks];
  const void* gamma;
  size_t rows;
  size_t hidden;
  float eps;
};

template <int DT>
__device__ __forceinline__ void widen(uint4 v, float* f) {
  Acc a;
  acc_init<DT>(a, v);
#pragma unroll
  for (int i = 0; i < Elem<DT>::kPerUnit; ++i) f[i] = __uint_as_float(a.w[i]);
}

template <int N, int DT, bool VEC>
__global__ void __launch_bounds__(kNormThreads) allreduce_rmsnorm_kernel(const __grid_constant__ NormArgs a) {
  constexpr int PU = Elem<DT>::kPerUnit;
  constexpr int ES = Elem<DT>::kSize;
  extern __shared__ float srow[];  // hidden float32 sums (padded to whole units)
  __shared__ float s_part[kNormThreads / 32];
  const size_t hidden = a.hidden;
  const size_t units = (hidden + PU - 1) / PU;
  const size_t row_off = (size_t)blockIdx.x * hidden * ES;
  const int tid = threadIdx.x;

  float ss = 0.f;
  for (size_t u = tid; u < units; u += kNormThreads) {
    const int v = unit_valid<DT>(u, hidden);
    uint4 x[N];
#pragma unroll
    for (int k = 0; k < N; ++k) x[k] = load_in<DT, VEC>(static_cast<const char*>(a.in[k]) + row_off, u, v);
    Acc s;
    acc_init<DT>(s, x[0]);
#pragma unroll
    for (int k = 1; k < N; ++k) acc_add<DT>(s, x[k]);
#pragma unroll
    for (int i = 0; i < PU; ++i) {
      const float f = i < v ? __uint_as_float(s.w[i]) : 0.f;
      srow[u * PU + i] = f;
      ss = __fmaf_rn(f, f, ss);
    }
  }
  // block reduction of the sum of squares
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((tid & 31) == 0) s_part[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += s_part[w];
  const float inv = rsqrtf(tot / (float)hidden + a.eps);

  for (size_t u = tid; u < units; u += kNormThreads) {
    const int v = unit_valid<DT>(u, hidden);
    float g[PU];
    widen<DT>(load_in<DT, VEC>(a.gamma, u, v), g);
    Acc y;
#pragma unroll
    for (int i = 0; i < PU; ++i) y.w[i] = __float_as_uint(__fmul_rn(__fmul_rn(srow[u * PU + i], inv), g[i]));
    const uint4 o = acc_narrow<DT>(y);
#pragma unroll
    for (int r = 0; r < N; ++r) store_out<DT, VEC, true>(static_cast<char*>(a.out[r]) + row_off, u, v, o);
  }
}

template <int N, int DT, bool VEC>
static cudaError_t norm_go(const NormArgs& a, cudaStream_t s) {
  const size_t smem = ((a.hidden + 7) / 8) * 8 * sizeof(float);
  static const cudaError_t attr = cudaFuncSetAttribute(
      allreduce_rmsnorm_kernel<N, DT, VEC>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  if (attr != cudaSuccess) return attr;
  allreduce_rmsnorm_kernel<N, DT, VEC><<<(unsigned)a.rows, kNormThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <int N>
static cudaError_t norm_n(int dt, bool vec, const NormArgs& a, cudaStream_t s) {
  if (dt == RRA_FLOAT32) return vec ? norm_go<N, RRA_FLOAT32, true>(a, s) : norm_go<N, RRA_FLOAT32, false>(a, s);
  return vec ? norm_go<N, RRA_BFLOAT16, true>(a, s) : norm_go<N, RRA_BFLOAT16, false>(a, s);
}

cudaError_t launch_allreduce_rmsnorm(int n, int dt, bool vec, const void* const* in, void* const* out,
                                     const void* gamma, size_t rows, size_t hidden, float eps,
                                     cudaStream_t s) {
  NormArgs a{};
  for (int r = 0; r < n; ++r) {
    a.in[r] = in[r];
    a.out[r] = out[r];
  }
  a.gamma = gamma;
  a.rows = rows;
  a.hidden = hidden;
  a.eps = eps;
  switch (n) {
    case 1: return norm_n<1>(dt, vec, a, s);
    case 2: return norm_n<2>(dt, vec, a, s);
    case 3: return norm_n<3>(dt, vec, a, s);
    case 4: return norm_n<4>(dt, vec, a, s);
    case 5: return norm_n<5>(dt, vec, a, s);
    case 6: return norm_n<6>(dt, vec, a, s);
    case 7: return norm_n<7>(dt, vec, a, s);
    case 8: return norm_n<8>(dt, vec, a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace rra
