// common.cuh -- device helpers shared by the kernels: 16-byte unit I/O with
// cache hints, element types with float32 accumulation, flags with
// acquire/release semantics, bounded waits and the per-call epoch.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "rra_internal.h"

namespace rra {

// ---------------------------------------------------------------------------
// memory access
// ---------------------------------------------------------------------------

// Input read once per call: no L1 allocation (nothing reuses it in the SM).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Data written by another CTA of the same kernel: read at L2, never from a
// possibly stale L1 line.
__device__ __forceinline__ uint4 ld_l2(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// Final output: streaming store (evict first).
__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Output another CTA reads back soon (two-shot phase 1, FIFO slots).
__device__ __forceinline__ void st_l2(void* p, uint4 v) {
  asm volatile("st.global.cg.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Polled lines (LL, LL128): one 16-byte access, never cached in L1.
__device__ __forceinline__ uint4 ld_volatile(const void* p) {
  uint4 v;
  asm volatile("ld.volatile.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ void st_volatile(void* p, uint4 v) {
  asm volatile("st.volatile.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_volatile8(void* p, uint32_t a, uint32_t b) {
  asm volatile("st.volatile.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

// Two LL lines (8 bytes each: a 4-byte data word under a 4-byte flag) in
// one 16-byte access; each 8-byte line is single-copy atomic, so a reader
// that sees a line's flag sees its data.
__device__ __forceinline__ void st_ll_pair(void* p, uint32_t flag, uint32_t a, uint32_t b) {
  const unsigned long long x = ((unsigned long long)flag << 32) | a;
  const unsigned long long y = ((unsigned long long)flag << 32) | b;
  asm volatile("st.volatile.global.v2.u64 [%0], {%1,%2};" ::"l"(p), "l"(x), "l"(y) : "memory");
}

__device__ __forceinline__ void ld_ll_pair(const void* p, unsigned long long& x, unsigned long long& y) {
  asm volatile("ld.volatile.global.v2.u64 {%0,%1}, [%2];" : "=l"(x), "=l"(y) : "l"(p) : "memory");
}

__device__ __forceinline__ uint64_t ld_acquire(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void fence_acq_rel() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// element types.  A "unit" is 16 bytes: 4 int32 / float32 or 8 bfloat16.
// Accumulators: uint32 (int32, wraps mod 2^32) or float (float32, bfloat16).
// ---------------------------------------------------------------------------
template <int DT>
struct Elem;
template <>
struct Elem<RRA_INT32> {
  static constexpr int kSize = 4, kPerUnit = 4, kAccWords = 1;  // accumulator units per unit
};
template <>
struct Elem<RRA_FLOAT32> {
  static constexpr int kSize = 4, kPerUnit = 4, kAccWords = 1;
};
template <>
struct Elem<RRA_BFLOAT16> {
  static constexpr int kSize = 2, kPerUnit = 8, kAccWords = 2;
};

struct Acc {
  uint32_t w[8];  // int32: w[0..3]; float32: w[0..3] float bits; bfloat16: w[0..7] float bits
};

template <int DT>
__device__ __forceinline__ void acc_init(Acc& a, uint4 v) {
  if constexpr (DT == RRA_BFLOAT16) {
    const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      a.w[2 * i] = x[i] << 16;             // element 2i (low half) widened exactly
      a.w[2 * i + 1] = x[i] & 0xFFFF0000u;  // element 2i+1
    }
  } else {
    a.w[0] = v.x;
    a.w[1] = v.y;
    a.w[2] = v.z;
    a.w[3] = v.w;
  }
}

// a = a (+) v: the running sum first, the new operand second.
template <int DT>
__device__ __forceinline__ void acc_add(Acc& a, uint4 v) {
  if constexpr (DT == RRA_INT32) {
    a.w[0] += v.x;
    a.w[1] += v.y;
    a.w[2] += v.z;
    a.w[3] += v.w;
  } else if constexpr (DT == RRA_FLOAT32) {
    a.w[0] = __float_as_uint(__fadd_rn(__uint_as_float(a.w[0]), __uint_as_float(v.x)));
    a.w[1] = __float_as_uint(__fadd_rn(__uint_as_float(a.w[1]), __uint_as_float(v.y)));
    a.w[2] = __float_as_uint(__fadd_rn(__uint_as_float(a.w[2]), __uint_as_float(v.z)));
    a.w[3] = __float_as_uint(__fadd_rn(__uint_as_float(a.w[3]), __uint_as_float(v.w)));
  } else {
    const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      a.w[2 * i] =
          __float_as_uint(__fadd_rn(__uint_as_float(a.w[2 * i]), __uint_as_float(x[i] << 16)));
      a.w[2 * i + 1] = __float_as_uint(
          __fadd_rn(__uint_as_float(a.w[2 * i + 1]), __uint_as_float(x[i] & 0xFFFF0000u)));
    }
  }
}

// Round the accumulator to the element type (bfloat16: nearest even, by the
// CUDA conversion intrinsic).
template <int DT>
__device__ __forceinline__ uint4 acc_narrow(const Acc& a) {
  if constexpr (DT == RRA_BFLOAT16) {
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h =
          __floats2bfloat162_rn(__uint_as_float(a.w[2 * i]), __uint_as_float(a.w[2 * i + 1]));
      o[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  } else {
    return make_uint4(a.w[0], a.w[1], a.w[2], a.w[3]);
  }
}

// Accumulator <-> FIFO words (ring partial sums keep float32 for bfloat16).
template <int DT>
__device__ __forceinline__ void acc_to_words(const Acc& a, uint4* w) {
  w[0] = make_uint4(a.w[0], a.w[1], a.w[2], a.w[3]);
  if constexpr (Elem<DT>::kAccWords == 2) w[1] = make_uint4(a.w[4], a.w[5], a.w[6], a.w[7]);
}

template <int DT>
__device__ __forceinline__ void acc_from_words(Acc& a, const uint4* w) {
  a.w[0] = w[0].x;
  a.w[1] = w[0].y;
  a.w[2] = w[0].z;
  a.w[3] = w[0].w;
  if constexpr (Elem<DT>::kAccWords == 2) {
    a.w[4] = w[1].x;
    a.w[5] = w[1].y;
    a.w[6] = w[1].z;
    a.w[7] = w[1].w;
  }
}

// ---------------------------------------------------------------------------
// unit I/O with a partial last unit and an element-wise path for buffers
// that are not 16-byte aligned.  `valid` = elements of the unit in range.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ uint4 ld_partial(const char* p, int valid) {
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  if constexpr (Elem<DT>::kSize == 4) {
    for (int i = 0; i < valid; ++i) w[i] = __ldg(reinterpret_cast<const unsigned int*>(p) + i);
  } else {
    for (int i = 0; i < valid; ++i)
      w[i >> 1] |= (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p) + i) << (16 * (i & 1));
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int DT>
__device__ __forceinline__ uint4 ld_partial_l2(const char* p, int valid) {
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  if constexpr (Elem<DT>::kSize == 4) {
    for (int i = 0; i < valid; ++i) w[i] = __ldcg(reinterpret_cast<const unsigned int*>(p) + i);
  } else {
    for (int i = 0; i < valid; ++i)
      w[i >> 1] |= (uint32_t)__ldcg(reinterpret_cast<const unsigned short*>(p) + i) << (16 * (i & 1));
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int DT>
__device__ __forceinline__ void st_partial(char* p, uint4 v, int valid) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if constexpr (Elem<DT>::kSize == 4) {
    for (int i = 0; i < valid; ++i) reinterpret_cast<unsigned int*>(p)[i] = w[i];
  } else {
    for (int i = 0; i < valid; ++i)
      reinterpret_cast<unsigned short*>(p)[i] = (unsigned short)(w[i >> 1] >> (16 * (i & 1)));
  }
}

// Load unit u of `base` (a read-only input).
template <int DT, bool VEC>
__device__ __forceinline__ uint4 load_in(const void* base, size_t u, int valid) {
  const char* p = static_cast<const char*>(base) + u * 16;
  if (VEC && valid == Elem<DT>::kPerUnit) return ld_stream(p);
  return ld_partial<DT>(p, valid);
}

// Load unit u of a buffer another CTA wrote in this kernel.
template <int DT, bool VEC>
__device__ __forceinline__ uint4 load_shared_out(const void* base, size_t u, int valid) {
  const char* p = static_cast<const char*>(base) + u * 16;
  if (VEC && valid == Elem<DT>::kPerUnit) return ld_l2(p);
  return ld_partial_l2<DT>(p, valid);
}

template <int DT, bool VEC, bool STREAM>
__device__ __forceinline__ void store_out(void* base, size_t u, int valid, uint4 v) {
  char* p = static_cast<char*>(base) + u * 16;
  if (VEC && valid == Elem<DT>::kPerUnit) {
    if (STREAM)
      st_stream(p, v);
    else
      st_l2(p, v);
  } else {
    st_partial<DT>(p, v, valid);
  }
}

template <int DT>
__device__ __forceinline__ int unit_valid(size_t u, size_t count) {
  constexpr int PU = Elem<DT>::kPerUnit;
  const size_t lo = u * PU;
  return lo + PU <= count ? PU : (lo < count ? (int)(count - lo) : 0);
}

// ---------------------------------------------------------------------------
// epoch, bounded waits, errors
// ---------------------------------------------------------------------------
constexpr uint32_t kMaxSpin = 1u << 26;  // backstop iteration cap on every wait

__device__ __forceinline__ void record_error(DevStatus* st, int code, int rank, int peer, int index,
                                             uint32_t tag, bool root = false) {
  const unsigned long long d = (1ull << 63) | ((unsigned long long)(index & 0x7FFFFFFF) << 32) |
                               ((unsigned long long)(peer & 0xFFFF) << 16) |
                               (unsigned long long)(rank & 0xFFFF);
  atomicCAS(&st->code, 0, code);
  atomicCAS(&st->detail, 0ull, d);
  if (root) atomicExch(&st->root_detail, d);
  atomicExch(&st->abort_tag, tag);
}

__device__ __forceinline__ bool aborted(const DevStatus* st, uint32_t tag) {
  return ld_relaxed_u32(&st->abort_tag) == tag;
}

// Wait until *flag >= target; *seen gets the value observed.  Returns false
// (after recording a timeout unless another wait already gave up) when the
// wait expires or the call was aborted.  Never unbounded: a %globaltimer
// limit plus an iteration cap.  An expired wait is the "root" record when
// the peer never joined the call: by default when the awaited flag itself
// holds an earlier call's value; with `joined`, when the peer's joined flag
// (raised by each of its CTAs before any wait) does.
static __device__ __noinline__ bool wait_geq(const uint64_t* flag, uint64_t target, uint64_t* seen,
                                      const WaitCfg& w, uint32_t tag, int rank, int peer,
                                      int index, const uint64_t* joined = nullptr) {
  uint64_t v = ld_acquire(flag);
  if (v >= target) {
    *seen = v;
    return true;
  }
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1; it < kMaxSpin; ++it) {
    v = ld_acquire(flag);
    if (v >= target) {
      *seen = v;
      return true;
    }
    if ((it & 15u) == 0u) {
      if (aborted(w.status, tag)) return false;
      if (globaltimer() - t0 > w.timeout_ns) break;
    }
    __nanosleep(64);
  }
  // The flag (or the peer's joined flag) still holds a value of an earlier
  // call: the peer took no part in this one.
  const bool root = joined ? (ld_acquire(joined) >> 32) != (target >> 32) : (v >> 32) != (target >> 32);
  record_error(w.status, RRA_ERR_TIMEOUT, rank, peer, index, tag, root);
  return false;
}

// Every CTA of a synchronizing kernel reads the call epoch first; flags of
// this call carry (epoch << 32) | count, so values left by earlier calls
// compare lower and no flag needs resetting.
__device__ __forceinline__ uint32_t read_epoch(SyncHdr* s) { return ld_relaxed_u32(&s->epoch); }

// The last CTA to finish bumps the epoch.  The next kernel on the stream
// starts after this one has ended, so it sees the new epoch.
__device__ __forceinline__ void arrive_end(SyncHdr* s, uint32_t epoch) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t total = gridDim.x * gridDim.y * gridDim.z;
    const uint32_t old = atomicAdd(&s->arrive, 1u);
    if (old == total - 1u) {
      atomicExch(&s->arrive, 0u);
      atomicExch(&s->epoch, epoch + 1u);
    }
  }
}

}  // namespace rra
