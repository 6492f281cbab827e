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
// is zero-padded.  A line is always written by one aligned store at least
// as wide as the line part it carries (16-byte stores holding two LL lines,
// or a 16-byte part of an LL128 line), so a reader that sees the flag sees
// the data stored with it.  LL128's guarantee for whole 128-byte lines is
// an NVLink property; here a warp checks all four flags of its four lines
// before it uses any of their data.
#include "common.cuh"

namespace rra {

// ---------------------------------------------------------------------------
// LL
// ---------------------------------------------------------------------------

// Thread g packs payload bytes [16g, 16g+16) into lines 4g..4g+3.
__global__ void __launch_bounds__(kLLThreads) ll_pack_kernel(const __grid_constant__ LLArgs a) {
  const size_t B = a.payload_bytes;
  const size_t lines = (B + 3) / 4;
  const size_t groups = (lines + 3) / 4;
  const uint32_t f = (uint32_t)a.flag;
  const unsigned char* p = static_cast<const unsigned char*>(a.payload);
  char* wire = static_cast<char*>(a.wire_out);
  for (size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x; g < groups;
       g += (size_t)gridDim.x * blockDim.x) {
    const size_t off = g * 16;
    uint4 v;
    if (a.vec && off + 16 <= B) {
      v = ld_stream(p + off);
    } else {
      uint32_t w[4] = {0u, 0u, 0u, 0u};
      for (int b = 0; b < 16 && off + b < B; ++b) w[b >> 2] |= (uint32_t)__ldg(p + off + b) << (8 * (b & 3));
      v = make_uint4(w[0], w[1], w[2], w[3]);
    }
    const size_t nl = lines - 4 * g < 4 ? lines - 4 * g : 4;
    char* w = wire + g * 32;
    if (nl >= 2)
      st_volatile(w, make_uint4(v.x, f, v.y, f));
    else
      st_volatile8(w, v.x, f);
    if (nl == 4)
      st_volatile(w + 16, make_uint4(v.z, f, v.w, f));
    else if (nl == 3)
      st_volatile8(w + 16, v.z, f);
  }
}

__device__ __forceinline__ uint2 ld_volatile8(const void* p) {
  uint2 v;
  asm volatile("ld.volatile.global.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p) : "memory");
  return v;
}

// Lines 4g..4g+3 of one wire: data words and whether every present line's
// flag equals `want`.
__device__ __forceinline__ bool ll_read4(const char* w, size_t nl, uint32_t want, uint32_t d[4]) {
  uint32_t fl[4] = {want, want, want, want};
  if (nl >= 2) {
    const uint4 a = ld_volatile(w);
    d[0] = a.x; fl[0] = a.y; d[1] = a.z; fl[1] = a.w;
  } else {
    const uint2 a = ld_volatile8(w);
    d[0] = a.x; fl[0] = a.y; d[1] = 0u;
  }
  if (nl == 4) {
    const uint4 b = ld_volatile(w + 16);
    d[2] = b.x; fl[2] = b.y; d[3] = b.z; fl[3] = b.w;
  } else if (nl == 3) {
    const uint2 b = ld_volatile8(w + 16);
    d[2] = b.x; fl[2] = b.y; d[3] = 0u;
  } else {
    d[2] = 0u; d[3] = 0u;
  }
  return fl[0] == want && fl[1] == want && fl[2] == want && fl[3] == want;
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
  for (size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x; g < groups;
       g += (size_t)gridDim.x * blockDim.x) {
    const size_t nl = lines - 4 * g < 4 ? lines - 4 * g : 4;
    uint32_t d[NSRC][4];
    bool stop = false;
#pragma unroll
    for (int k = 0; k < NSRC; ++k) {
      const char* w = static_cast<const char*>(a.wire_in[k]) + g * 32;
      if (!ll_read4(w, nl, want, d[k])) {
        // bounded poll until the line's flags arrive
        const uint64_t t0 = globaltimer();
        bool ok = false;
        for (uint32_t it = 0; it < kMaxSpin; ++it) {
          __nanosleep(64);
          if (ll_read4(w, nl, want, d[k])) { ok = true; break; }
          if ((it & 15u) == 15u) {
            if (aborted(a.wait.status, tag)) break;
            if (globaltimer() - t0 > a.wait.timeout_ns) {
              // name the first present line of the group whose flag differs
              int bad = 0;
              for (int i = 0; i < (int)nl; ++i) {
                const uint32_t fi = *reinterpret_cast<const volatile uint32_t*>(w + 8 * i + 4);
                if (fi != want) { bad = i; break; }
              }
              record_error(a.wait.status, RRA_ERR_TIMEOUT, k, -1, (int)(4 * g + bad), tag);
              break;
            }
          }
        }
        if (!ok) { stop = true; break; }
      }
    }
    if (stop) break;
    Acc s;
    acc_init<DT>(s, make_uint4(d[0][0], d[0][1], d[0][2], d[0][3]));
#pragma unroll
    for (int k = 1; k < NSRC; ++k) acc_add<DT>(s, make_uint4(d[k][0], d[k][1], d[k][2], d[k][3]));
    const uint4 y = acc_narrow<DT>(s);
    const size_t off = g * 16;
    if (a.vec && off + 16 <= B) {
      st_stream(out + off, y);
    } else {
      const uint32_t w[4] = {y.x, y.y, y.z, y.w};
      for (int b = 0; b < 16 && off + b < B; ++b) out[off + b] = (char)(w[b >> 2] >> (8 * (b & 3)));
    }
  }
  arrive_end(a.wait.sync, epoch);
}

// ---------------------------------------------------------------------------
// LL128: a warp handles four lines; lane l covers bytes [16(l%8), +16) of
// line 4q + l/8; lanes 7, 15, 23, 31 carry the line's 8 data bytes and flag.
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
  for (size_t q = (size_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); q < quads; q += warps) {
    const size_t j = 4 * q + (lane >> 3);
    if (j >= lines) continue;
    const size_t off = 120 * j + 16 * li;  // 8-byte aligned
    const int nbytes = li < 7 ? 16 : 8;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (a.vec && off + nbytes <= B) {
      const uint2 lo = ld_nc8(p + off);
      w[0] = lo.x;
      w[1] = lo.y;
      if (li < 7) {
        const uint2 hi = ld_nc8(p + off + 8);
        w[2] = hi.x;
        w[3] = hi.y;
      }
    } else {
      for (int b = 0; b < nbytes && off + b < B; ++b) w[b >> 2] |= (uint32_t)__ldg(p + off + b) << (8 * (b & 3));
    }
    if (li == 7) {
      w[2] = (uint32_t)a.flag;
      w[3] = (uint32_t)(a.flag >> 32);
    }
    st_volatile(wire + 128 * j + 16 * li, make_uint4(w[0], w[1], w[2], w[3]));
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
  for (size_t q = (size_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); q < quads; q += warps) {
    const size_t j = 4 * q + (lane >> 3);
    const bool present = j < lines;
    uint4 v[NSRC];
    bool stop = false;
#pragma unroll
    for (int k = 0; k < NSRC; ++k) {
      const char* w = static_cast<const char*>(a.wire_in[k]) + 128 * j + 16 * li;
      uint64_t t0 = 0;
      for (uint32_t it = 0;; ++it) {
        v[k] = present ? ld_volatile(w) : make_uint4(0u, 0u, 0u, 0u);
        const bool mine = li != 7 || !present ||
                          ((uint64_t)v[k].z | ((uint64_t)v[k].w << 32)) == want;
        // the flag lane of each line tells the line's lanes; then the warp agrees
        const bool line_ok = __shfl_sync(0xffffffffu, mine, lane | 7);
        if (__all_sync(0xffffffffu, line_ok)) break;
        if (it == 0) t0 = globaltimer();
        int give_up = 0;
        if (lane == 0 && (it & 15u) == 15u) {
          if (aborted(a.wait.status, tag)) give_up = 1;
          else if (globaltimer() - t0 > a.wait.timeout_ns || it >= kMaxSpin) give_up = 2;
        }
        give_up = __shfl_sync(0xffffffffu, give_up, 0);
        if (give_up) {
          const unsigned bad = __ballot_sync(0xffffffffu, !line_ok);
          if (give_up == 2 && lane == 0)
            record_error(a.wait.status, RRA_ERR_TIMEOUT, k, -1, (int)(4 * q + (__ffs(bad) - 1) / 8), tag);
          stop = true;
          break;
        }
        __nanosleep(64);
      }
      if (stop) break;
    }
    if (stop) break;
    Acc s;
    acc_init<DT>(s, v[0]);
#pragma unroll
    for (int k = 1; k < NSRC; ++k) acc_add<DT>(s, v[k]);
    const uint4 y = acc_narrow<DT>(s);
    if (!present) continue;
    const size_t off = 120 * j + 16 * li;
    const int nbytes = li < 7 ? 16 : 8;
    if (a.vec && off + nbytes <= B) {
      uint2* o = reinterpret_cast<uint2*>(out + off);  // 8-byte aligned
      o[0] = make_uint2(y.x, y.y);
      if (li < 7) o[1] = make_uint2(y.z, y.w);
    } else {
      const uint32_t w[4] = {y.x, y.y, y.z, y.w};
      for (int b = 0; b < nbytes && off + b < B; ++b) out[off + b] = (char)(w[b >> 2] >> (8 * (b & 3)));
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
