// kernels_ll.cu -- LL and LL128 wire formats: pack, and unpack fused with
// a SUM over several sources.
//
// "Collective communication: NCCL's algorithms and protocols, and custom
// all-reduce in inference frameworks", section "Protocols: how do you know
// the data has arrived":
//   LL    -- every 8 bytes hold 4 bytes of data and 4 bytes of flag; the
//            receiver polls the flag; relies on 8-byte writes being atomic,
//            so no memory fence is needed (about 50% efficiency);
//   LL128 -- every 128 bytes hold 120 bytes of data and 8 bytes of flag
//            (about 94% efficiency).
// Layout used here: data first, flag last, little-endian; the payload's tail
// is zero-padded.
//
// LL lines are written and read as 64-bit elements (two per 16-byte vector
// access), and an aligned 64-bit access is single-copy atomic, so a reader
// that sees a line's flag sees the data stored with it.  LL128's guarantee
// for whole 128-byte lines is an NVLink property with no equivalent inside
// one GPU; the LL128 kernels here are exact in stream order (pack, then
// unpack on the same or an ordered stream) and check every line's flag, but
// a reader running concurrently with the writer could see a flag before
// the rest of its line.
//
// Throughput: every thread (LL) or warp (LL128) keeps several line groups
// in flight per trip of its grid-stride loop.
#include "common.cuh"

namespace rra {

constexpr int kLLUnroll = 4;    // 16-byte payload groups per thread per trip (LL)
constexpr int kL128Unroll = 2;  // four-line quads per warp per trip (LL128)

__device__ __forceinline__ unsigned long long ll_line(uint32_t data, uint32_t flag) {
  return ((unsigned long long)flag << 32) | data;
}

__device__ __forceinline__ void st_lines2(void* p, unsigned long long a, unsigned long long b) {
  asm volatile("st.volatile.global.v2.u64 [%0], {%1,%2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}

__device__ __forceinline__ void st_line1(void* p, unsigned long long a) {
  asm volatile("st.volatile.global.u64 [%0], %1;" ::"l"(p), "l"(a) : "memory");
}

__device__ __forceinline__ void ld_lines2(const void* p, unsigned long long& a, unsigned long long& b) {
  asm volatile("ld.volatile.global.v2.u64 {%0,%1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

__device__ __forceinline__ unsigned long long ld_line1(const void* p) {
  unsigned long long a;
  asm volatile("ld.volatile.global.u64 %0, [%1];" : "=l"(a) : "l"(p) : "memory");
  return a;
}

// payload bytes [off, off+16), zero past B
__device__ __forceinline__ uint4 load_payload16(const unsigned char* p, size_t off, size_t B, bool vec) {
  if (vec && off + 16 <= B) return ld_stream(p + off);
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  for (int b = 0; b < 16 && off + b < B; ++b) w[b >> 2] |= (uint32_t)__ldg(p + off + b) << (8 * (b & 3));
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// ---------------------------------------------------------------------------
// LL: group g = payload bytes [16g, 16g+16) = lines 4g..4g+3 = wire bytes
// [32g, 32g+32)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kLLThreads) ll_pack_kernel(const __grid_constant__ LLArgs a) {
  const size_t B = a.payload_bytes;
  const size_t lines = (B + 3) / 4;
  const size_t groups = (lines + 3) / 4;
  const uint32_t f = (uint32_t)a.flag;
  const unsigned char* p = static_cast<const unsigned char*>(a.payload);
  char* wire = static_cast<char*>(a.wire_out);
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t g0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x; g0 < groups; g0 += kLLUnroll * stride) {
    uint4 v[kLLUnroll];
#pragma unroll
    for (int k = 0; k < kLLUnroll; ++k) {
      const size_t g = g0 + k * stride;
      if (g < groups) v[k] = load_payload16(p, g * 16, B, a.vec);
    }
#pragma unroll
    for (int k = 0; k < kLLUnroll; ++k) {
      const size_t g = g0 + k * stride;
      if (g >= groups) continue;
      const size_t nl = lines - 4 * g < 4 ? lines - 4 * g : 4;
      char* w = wire + g * 32;
      if (nl >= 2)
        st_lines2(w, ll_line(v[k].x, f), ll_line(v[k].y, f));
      else
        st_line1(w, ll_line(v[k].x, f));
      if (nl == 4)
        st_lines2(w + 16, ll_line(v[k].z, f), ll_line(v[k].w, f));
      else if (nl == 3)
        st_line1(w + 16, ll_line(v[k].z, f));
    }
  }
}

// Lines 4g..4g+3 of one wire: data words and whether every present line's
// flag equals `want`.
__device__ __forceinline__ bool ll_read4(const char* w, size_t nl, uint32_t want, uint32_t d[4]) {
  unsigned long long l[4] = {0ull, 0ull, 0ull, 0ull};
  if (nl >= 2)
    ld_lines2(w, l[0], l[1]);
  else
    l[0] = ld_line1(w);
  if (nl == 4)
    ld_lines2(w + 16, l[2], l[3]);
  else if (nl == 3)
    l[2] = ld_line1(w + 16);
  bool ok = true;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    d[i] = (uint32_t)l[i];
    if ((size_t)i < nl) ok = ok && (uint32_t)(l[i] >> 32) == want;
  }
  return ok;
}

template <int DT, int NSRC>
__global__ void __launch_bounds__(kLLThreads) ll_unpack_kernel(const __grid_constant__ LLArgs a) {
  __shared__ uint32_t s_epoch;
  if (threadIdx.x == 0) s_epoch = read_epoch(a.wait.sync);
  __syncthreads();
  const uint32_t epoch = s_epoch, tag = epoch + 1u;
  const size_t B = a.payload_bytes;
  const size_t lines = (B + 3) / 4;
  const size_t groups = (lines + 3) / 4;
  const uint32_t want = (uint32_t)a.flag;
  char* out = static_cast<char*>(a.out);
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  bool stop = false;
  for (size_t g0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x; g0 < groups && !stop;
       g0 += kLLUnroll * stride) {
    uint32_t d[kLLUnroll][NSRC][4];
    bool ok[kLLUnroll][NSRC];
    // first pass: every line of every source in flight at once
#pragma unroll
    for (int k = 0; k < kLLUnroll; ++k) {
      const size_t g = g0 + k * stride;
      if (g >= groups) continue;
      const size_t nl = lines - 4 * g < 4 ? lines - 4 * g : 4;
#pragma unroll
      for (int s = 0; s < NSRC; ++s)
        ok[k][s] = ll_read4(static_cast<const char*>(a.wire_in[s]) + g * 32, nl, want, d[k][s]);
    }
#pragma unroll
    for (int k = 0; k < kLLUnroll; ++k) {
      const size_t g = g0 + k * stride;
      if (g >= groups || stop) continue;
      const size_t nl = lines - 4 * g < 4 ? lines - 4 * g : 4;
#pragma unroll
      for (int s = 0; s < NSRC; ++s) {
        if (ok[k][s] || stop) continue;
        // bounded poll until the line's flags arrive
        const char* w = static_cast<const char*>(a.wire_in[s]) + g * 32;
        const uint64_t t0 = globaltimer();
        bool got = false;
        for (uint32_t it = 0; it < kMaxSpin; ++it) {
          __nanosleep(64);
          if (ll_read4(w, nl, want, d[k][s])) {
            got = true;
            break;
          }
          if ((it & 15u) == 15u) {
            if (aborted(a.wait.status, tag)) break;
            if (globaltimer() - t0 > a.wait.timeout_ns) {
              int bad = 0;  // first present line of the group whose flag differs
              for (int i = 0; i < (int)nl; ++i)
                if ((uint32_t)(ld_line1(w + 8 * i) >> 32) != want) {
                  bad = i;
                  break;
                }
              record_error(a.wait.status, RRA_ERR_TIMEOUT, s, -1, (int)(4 * g + bad), tag);
              break;
            }
          }
        }
        if (!got) stop = true;
      }
      if (stop) continue;
      Acc acc;
      acc_init<DT>(acc, make_uint4(d[k][0][0], d[k][0][1], d[k][0][2], d[k][0][3]));
#pragma unroll
      for (int s = 1; s < NSRC; ++s)
        acc_add<DT>(acc, make_uint4(d[k][s][0], d[k][s][1], d[k][s][2], d[k][s][3]));
      const uint4 y = acc_narrow<DT>(acc);
      const size_t off = g * 16;
      if (a.vec && off + 16 <= B) {
        st_stream(out + off, y);
      } else {
        const uint32_t w[4] = {y.x, y.y, y.z, y.w};
        for (int b = 0; b < 16 && off + b < B; ++b) out[off + b] = (char)(w[b >> 2] >> (8 * (b & 3)));
      }
    }
  }
  arrive_end(a.wait.sync, epoch);
}

// ---------------------------------------------------------------------------
// LL128: a warp handles four lines (a quad); lane l covers bytes
// [16(l%8), +16) of line 4q + l/8; lanes 7, 15, 23, 31 carry the line's
// last 8 data bytes and its flag.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint2 ld_nc8(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__global__ void __launch_bounds__(kLLThreads) ll128_pack_kernel(const __grid_constant__ LLArgs a) {
  const size_t B = a.payload_bytes;
  const size_t lines = (B + 119) / 120;
  const size_t quads = (lines + 3) / 4;
  const int lane = threadIdx.x & 31, li = lane & 7;
  const size_t warps = (size_t)gridDim.x * (blockDim.x >> 5);
  const unsigned char* p = static_cast<const unsigned char*>(a.payload);
  char* wire = static_cast<char*>(a.wire_out);
  const int nbytes = li < 7 ? 16 : 8;
  for (size_t q0 = (size_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); q0 < quads;
       q0 += kL128Unroll * warps) {
    uint32_t w[kL128Unroll][4];
#pragma unroll
    for (int k = 0; k < kL128Unroll; ++k) {
      const size_t j = 4 * (q0 + k * warps) + (lane >> 3);
      w[k][0] = w[k][1] = w[k][2] = w[k][3] = 0u;
      if (j >= lines) continue;
      const size_t off = 120 * j + 16 * li;  // 8-byte aligned
      if (a.vec && off + nbytes <= B) {
        const uint2 lo = ld_nc8(p + off);
        w[k][0] = lo.x;
        w[k][1] = lo.y;
        if (li < 7) {
          const uint2 hi = ld_nc8(p + off + 8);
          w[k][2] = hi.x;
          w[k][3] = hi.y;
        }
      } else {
        for (int b = 0; b < nbytes && off + b < B; ++b)
          w[k][b >> 2] |= (uint32_t)__ldg(p + off + b) << (8 * (b & 3));
      }
    }
#pragma unroll
    for (int k = 0; k < kL128Unroll; ++k) {
      const size_t j = 4 * (q0 + k * warps) + (lane >> 3);
      if (j >= lines) continue;
      if (li == 7) {
        w[k][2] = (uint32_t)a.flag;
        w[k][3] = (uint32_t)(a.flag >> 32);
      }
      st_volatile(wire + 128 * j + 16 * li, make_uint4(w[k][0], w[k][1], w[k][2], w[k][3]));
    }
  }
}

template <int DT, int NSRC>
__global__ void __launch_bounds__(kLLThreads) ll128_unpack_kernel(const __grid_constant__ LLArgs a) {
  __shared__ uint32_t s_epoch;
  if (threadIdx.x == 0) s_epoch = read_epoch(a.wait.sync);
  __syncthreads();
  const uint32_t epoch = s_epoch, tag = epoch + 1u;
  const size_t B = a.payload_bytes;
  const size_t lines = (B + 119) / 120;
  const size_t quads = (lines + 3) / 4;
  const int lane = threadIdx.x & 31, li = lane & 7;
  const size_t warps = (size_t)gridDim.x * (blockDim.x >> 5);
  char* out = static_cast<char*>(a.out);
  const uint64_t want = a.flag;
  const int nbytes = li < 7 ? 16 : 8;
  for (size_t q0 = (size_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); q0 < quads;
       q0 += kL128Unroll * warps) {
    uint4 v[kL128Unroll][NSRC];
    bool present[kL128Unroll];
    // every line of every source in flight at once
#pragma unroll
    for (int k = 0; k < kL128Unroll; ++k) {
      const size_t j = 4 * (q0 + k * warps) + (lane >> 3);
      present[k] = (q0 + k * warps) < quads && j < lines;
#pragma unroll
      for (int s = 0; s < NSRC; ++s)
        v[k][s] = present[k] ? ld_volatile(static_cast<const char*>(a.wire_in[s]) + 128 * j + 16 * li)
                             : make_uint4(0u, 0u, 0u, 0u);
    }
    bool stop = false;
#pragma unroll
    for (int k = 0; k < kL128Unroll; ++k) {
      const size_t j = 4 * (q0 + k * warps) + (lane >> 3);
#pragma unroll
      for (int s = 0; s < NSRC; ++s) {
        const char* w = static_cast<const char*>(a.wire_in[s]) + 128 * j + 16 * li;
        uint64_t t0 = 0;
        for (uint32_t it = 0;; ++it) {
          const bool mine = li != 7 || !present[k] ||
                            ((uint64_t)v[k][s].z | ((uint64_t)v[k][s].w << 32)) == want;
          // the flag lane of each line tells the line's lanes; then the warp agrees
          const bool line_ok = __shfl_sync(0xffffffffu, mine, lane | 7);
          if (__all_sync(0xffffffffu, line_ok)) break;
          if (it == 0) t0 = globaltimer();
          int give_up = 0;
          if (lane == 0 && (it & 15u) == 15u) {
            if (aborted(a.wait.status, tag))
              give_up = 1;
            else if (globaltimer() - t0 > a.wait.timeout_ns || it >= kMaxSpin)
              give_up = 2;
          }
          give_up = __shfl_sync(0xffffffffu, give_up, 0);
          if (give_up) {
            const unsigned bad = __ballot_sync(0xffffffffu, !line_ok);
            if (give_up == 2 && lane == 0)
              record_error(a.wait.status, RRA_ERR_TIMEOUT, s, -1,
                           (int)(4 * (q0 + k * warps) + (__ffs(bad) - 1) / 8), tag);
            stop = true;
            break;
          }
          __nanosleep(64);
          if (present[k]) v[k][s] = ld_volatile(w);
        }
        if (stop) break;
      }
      if (stop) break;
    }
    if (stop) break;
#pragma unroll
    for (int k = 0; k < kL128Unroll; ++k) {
      if (!present[k]) continue;
      const size_t j = 4 * (q0 + k * warps) + (lane >> 3);
      Acc acc;
      acc_init<DT>(acc, v[k][0]);
#pragma unroll
      for (int s = 1; s < NSRC; ++s) acc_add<DT>(acc, v[k][s]);
      const uint4 y = acc_narrow<DT>(acc);
      const size_t off = 120 * j + 16 * li;
      if (a.vec && off + nbytes <= B) {
        uint2* o = reinterpret_cast<uint2*>(out + off);  // 8-byte aligned
        o[0] = make_uint2(y.x, y.y);
        if (li < 7) o[1] = make_uint2(y.z, y.w);
      } else {
        const uint32_t w[4] = {y.x, y.y, y.z, y.w};
        for (int b = 0; b < nbytes && off + b < B; ++b) out[off + b] = (char)(w[b >> 2] >> (8 * (b & 3)));
      }
    }
  }
  arrive_end(a.wait.sync, epoch);
}

// ---------------------------------------------------------------------------
// dispatch
// ---------------------------------------------------------------------------
cudaError_t launch_ll_pack(const LLArgs& a, int grid, cudaStream_t s) {
  ll_pack_kernel<<<grid, kLLThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_ll128_pack(const LLArgs& a, int grid, cudaStream_t s) {
  ll128_pack_kernel<<<grid, kLLThreads, 0, s>>>(a);
  return cudaGetLastError();
}

#define RRA_UNPACK_DISPATCH(KERNEL)                                                          \
  template <int DT>                                                                          \
  static cudaError_t KERNEL##_dt(const LLArgs& a, int grid, cudaStream_t s) {                \
    switch (a.nsrc) {                                                                        \
      case 1: KERNEL<DT, 1><<<grid, kLLThreads, 0, s>>>(a); break;                          \
      case 2: KERNEL<DT, 2><<<grid, kLLThreads, 0, s>>>(a); break;                          \
      case 3: KERNEL<DT, 3><<<grid, kLLThreads, 0, s>>>(a); break;                          \
      case 4: KERNEL<DT, 4><<<grid, kLLThreads, 0, s>>>(a); break;                          \
      case 5: KERNEL<DT, 5><<<grid, kLLThreads, 0, s>>>(a); break;                          \
      case 6: KERNEL<DT, 6><<<grid, kLLThreads, 0, s>>>(a); break;                          \
      case 7: KERNEL<DT, 7><<<grid, kLLThreads, 0, s>>>(a); break;                          \
      case 8: KERNEL<DT, 8><<<grid, kLLThreads, 0, s>>>(a); break;                          \
      default: return cudaErrorInvalidValue;                                                 \
    }                                                                                        \
    return cudaGetLastError();                                                               \
  }

RRA_UNPACK_DISPATCH(ll_unpack_kernel)
RRA_UNPACK_DISPATCH(ll128_unpack_kernel)

cudaError_t launch_ll_unpack(int dt, const LLArgs& a, int grid, cudaStream_t s) {
  if (dt == RRA_INT32) return ll_unpack_kernel_dt<RRA_INT32>(a, grid, s);
  if (dt == RRA_FLOAT32) return ll_unpack_kernel_dt<RRA_FLOAT32>(a, grid, s);
  return ll_unpack_kernel_dt<RRA_BFLOAT16>(a, grid, s);
}

cudaError_t launch_ll128_unpack(int dt, const LLArgs& a, int grid, cudaStream_t s) {
  if (dt == RRA_INT32) return ll128_unpack_kernel_dt<RRA_INT32>(a, grid, s);
  if (dt == RRA_FLOAT32) return ll128_unpack_kernel_dt<RRA_FLOAT32>(a, grid, s);
  return ll128_unpack_kernel_dt<RRA_BFLOAT16>(a, grid, s);
}

}  // namespace rra
