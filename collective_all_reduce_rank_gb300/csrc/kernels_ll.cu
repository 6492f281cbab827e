// kernels_ll.cu -- LL and LL128 wire formats: pack, and unpack fused with
// a SUM over several sources.
//
// The two formats are those of "Collective communication: NCCL's
// algorithms and protocols, and custom all-reduce in inference frameworks",
// section "Protocols: how do you know the data has arrived".  An LL line is
// 8 bytes, half payload and half flag, so it carries data at half the wire
// rate; the reader spins on the flag word, and since the 8 bytes travel in
// one indivisible store, finding the flag means finding the data, with no
// fence in between.  An LL128 line is 128 bytes: 120 of payload and an
// 8-byte flag, so 15/16 of the wire is data.  Layout used here: data first,
// flag last, little-endian; the payload's tail is zero-padded.
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
// Throughput: LL pack gives every thread one group of lines over a grid that
// covers the payload, LL128 pack eight quads per warp per trip (over a grid
// that covers the payload from 64 MiB); the unpack kernels keep several
// groups of every source in flight per thread, on a resident grid.  Partial groups
// and polling take out-of-line paths, so the fast paths stay lean.
#include "common.cuh"

namespace rra {

constexpr int kL128Unroll = 2;  // four-line quads per warp per trip (LL128 unpack)

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

__device__ __forceinline__ uint2 ld_nc8(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
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
// [32g, 32g+32).  Groups wholly inside the payload take a fast path with
// vector accesses only; the last, partial group (and every group of an
// unaligned payload) takes an out-of-line path, so the fast path keeps its
// registers and no local memory.
// ---------------------------------------------------------------------------
static __device__ __noinline__ void ll_pack_slow(const LLArgs& a, size_t g, size_t lines) {
  const size_t B = a.payload_bytes;
  const uint32_t f = (uint32_t)a.flag;
  const uint4 v = load_payload16(static_cast<const unsigned char*>(a.payload), g * 16, B, a.vec);
  const size_t nl = lines - 4 * g < 4 ? lines - 4 * g : 4;
  char* w = static_cast<char*>(a.wire_out) + g * 32;
  if (nl >= 2)
    st_lines2(w, ll_line(v.x, f), ll_line(v.y, f));
  else
    st_line1(w, ll_line(v.x, f));
  if (nl == 4)
    st_lines2(w + 16, ll_line(v.z, f), ll_line(v.w, f));
  else if (nl == 3)
    st_line1(w + 16, ll_line(v.z, f));
}

// One group per thread over a grid that covers the payload (the writes of a
// CTA stay together, which the wire, twice the payload, rewards).
__global__ void __launch_bounds__(kLLThreads) ll_pack_kernel(const __grid_constant__ LLArgs a) {
  const size_t B = a.payload_bytes;
  const size_t lines = (B + 3) / 4;
  const size_t groups = (lines + 3) / 4;
  const size_t full = a.vec ? B / 16 : 0;  // groups with all 16 payload bytes present
  const uint32_t f = (uint32_t)a.flag;
  const unsigned char* p = static_cast<const unsigned char*>(a.payload);
  char* wire = static_cast<char*>(a.wire_out);
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x; g < groups; g += stride) {
    if (g < full) {
      const uint4 v = ld_stream(p + g * 16);
      st_lines2(wire + g * 32, ll_line(v.x, f), ll_line(v.y, f));
      st_lines2(wire + g * 32 + 16, ll_line(v.z, f), ll_line(v.w, f));
    } else {
      ll_pack_slow(a, g, lines);
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

// Group g whose lines are not all there yet (or the partial last group):
// poll each source's lines, bounded, then sum in source order and store.
// False when a wait expired or the call was aborted.
template <int DT, int NSRC>
static __device__ __noinline__ bool ll_unpack_slow(const LLArgs& a, size_t g, size_t lines, uint32_t tag) {
  const size_t B = a.payload_bytes;
  const uint32_t want = (uint32_t)a.flag;
  const size_t nl = lines - 4 * g < 4 ? lines - 4 * g : 4;
  Acc acc;
  for (int s = 0; s < NSRC; ++s) {
    const char* w = static_cast<const char*>(a.wire_in[s]) + g * 32;
    uint32_t d[4];
    bool got = ll_read4(w, nl, want, d);
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 0; !got && it < kMaxSpin; ++it) {
      __nanosleep(64);
      got = ll_read4(w, nl, want, d);
      if (got) break;
      if ((it & 15u) == 15u) {
        if (aborted(a.wait.status, tag)) return false;
        if (globaltimer() - t0 > a.wait.timeout_ns) {
          int bad = 0;  // first present line of the group whose flag differs
          for (int i = 0; i < (int)nl; ++i)
            if ((uint32_t)(ld_line1(w + 8 * i) >> 32) != want) {
              bad = i;
              break;
            }
          record_error(a.wait.status, RRA_ERR_TIMEOUT, s, -1, (int)(4 * g + bad), tag);
          return false;
        }
      }
    }
    if (!got) return false;
    const uint4 v = make_uint4(d[0], d[1], d[2], d[3]);
    if (s == 0)
      acc_init<DT>(acc, v);
    else
      acc_add<DT>(acc, v);
  }
  const uint4 y = acc_narrow<DT>(acc);
  char* out = static_cast<char*>(a.out);
  const size_t off = g * 16;
  if (a.vec && off + 16 <= B) {
    st_stream(out + off, y);
  } else {
    const uint32_t w[4] = {y.x, y.y, y.z, y.w};
    for (int b = 0; b < 16 && off + b < B; ++b) out[off + b] = (char)(w[b >> 2] >> (8 * (b & 3)));
  }
  return true;
}

// groups per thread per trip: up to 8 source-groups (256 bytes of lines)
// in flight per thread, within the register budget of two CTAs per SM
template <int NSRC>
__host__ __device__ constexpr int ll_unpack_unroll() {
  return 8 / NSRC < 1 ? 1 : (8 / NSRC > 4 ? 4 : 8 / NSRC);
}

// Grid-stride over groups on a grid the GPU holds at once (so the per-call
// epoch costs one arrival per CTA); every line of every source of U groups
// is loaded before any flag is tested.
template <int DT, int NSRC>
__global__ void __launch_bounds__(kLLThreads, 2) ll_unpack_kernel(const __grid_constant__ LLArgs a) {
  constexpr int U = ll_unpack_unroll<NSRC>();
  __shared__ uint32_t s_epoch;
  if (threadIdx.x == 0) s_epoch = read_epoch(a.wait.sync);
  __syncthreads();
  const uint32_t epoch = s_epoch, tag = epoch + 1u;
  const size_t B = a.payload_bytes;
  const size_t lines = (B + 3) / 4;
  const size_t groups = (lines + 3) / 4;
  const size_t full = B / 16;
  const uint32_t want = (uint32_t)a.flag;
  char* out = static_cast<char*>(a.out);
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t g0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x; g0 < groups; g0 += U * stride) {
    unsigned long long l[U][NSRC][4];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const size_t g = g0 + k * stride;
      if (g < full) {
#pragma unroll
        for (int s = 0; s < NSRC; ++s) {
          const char* w = static_cast<const char*>(a.wire_in[s]) + g * 32;
          ld_lines2(w, l[k][s][0], l[k][s][1]);
          ld_lines2(w + 16, l[k][s][2], l[k][s][3]);
        }
      }
    }
    bool stop = false;
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const size_t g = g0 + k * stride;
      if (g >= groups) continue;
      bool ok = g < full && a.vec;
#pragma unroll
      for (int s = 0; s < NSRC; ++s)
#pragma unroll
        for (int i = 0; i < 4; ++i) ok = ok && (uint32_t)(l[k][s][i] >> 32) == want;
      if (ok) {
        Acc acc;
        acc_init<DT>(acc, make_uint4((uint32_t)l[k][0][0], (uint32_t)l[k][0][1], (uint32_t)l[k][0][2],
                                     (uint32_t)l[k][0][3]));
#pragma unroll
        for (int s = 1; s < NSRC; ++s)
          acc_add<DT>(acc, make_uint4((uint32_t)l[k][s][0], (uint32_t)l[k][s][1], (uint32_t)l[k][s][2],
                                      (uint32_t)l[k][s][3]));
        st_stream(out + g * 16, acc_narrow<DT>(acc));
      } else if (!ll_unpack_slow<DT, NSRC>(a, g, lines, tag)) {
        stop = true;
        break;
      }
    }
    if (stop) break;
  }
  arrive_end(a.wait.sync, epoch);
}

// ---------------------------------------------------------------------------
// LL128: a warp handles four lines (a quad); lane l covers bytes
// [16(l%8), +16) of line 4q + l/8; lanes 7, 15, 23, 31 carry the line's
// last 8 data bytes and its flag.
// ---------------------------------------------------------------------------

// Lane (line 4q + l/8, piece l%8) of a quad that is not complete, or of an
// unaligned payload: byte loads, zero past the payload's end.
static __device__ __noinline__ void ll128_pack_slow(const LLArgs& a, size_t j, int li) {
  const size_t B = a.payload_bytes;
  const unsigned char* p = static_cast<const unsigned char*>(a.payload);
  const int nbytes = li < 7 ? 16 : 8;
  const size_t off = 120 * j + 16 * li;
  uint32_t w0 = 0u, w1 = 0u, w2 = 0u, w3 = 0u;
  for (int b = 0; b < nbytes && off + b < B; ++b) {
    const uint32_t x = (uint32_t)__ldg(p + off + b) << (8 * (b & 3));
    if (b < 4)
      w0 |= x;
    else if (b < 8)
      w1 |= x;
    else if (b < 12)
      w2 |= x;
    else
      w3 |= x;
  }
  if (li == 7) {
    w2 = (uint32_t)a.flag;
    w3 = (uint32_t)(a.flag >> 32);
  }
  st_volatile(static_cast<char*>(a.wire_out) + 128 * j + 16 * li, make_uint4(w0, w1, w2, w3));
}


// kL128PackBatch quads per warp per trip of a grid-stride loop; whole quads
// of an aligned payload read their 120-byte line bodies with 8-byte loads
// (line j starts at byte 120j, a multiple of 8), every load of the trip
// issued before its stores.
__global__ void __launch_bounds__(kLLThreads) ll128_pack_kernel(const __grid_constant__ LLArgs a) {
  const size_t B = a.payload_bytes;
  const size_t lines = (B + 119) / 120;
  const size_t quads = (lines + 3) / 4;
  const size_t full = a.vec ? B / 480 : 0;  // quads whose four lines are complete
  const int lane = threadIdx.x & 31, li = lane & 7;
  const size_t warps = (size_t)gridDim.x * (blockDim.x >> 5);
  const unsigned char* p = static_cast<const unsigned char*>(a.payload);
  char* wire = static_cast<char*>(a.wire_out);
  const size_t q0 = (size_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  // whole quads: no call in the loop
  const uint2 flag2 = make_uint2((uint32_t)a.flag, (uint32_t)(a.flag >> 32));
  for (size_t q = q0; q < full; q += kL128PackBatch * warps) {
    uint2 lo[kL128PackBatch], hi[kL128PackBatch];
#pragma unroll
    for (int k = 0; k < kL128PackBatch; ++k) {
      const size_t qk = q + k * warps;
      const size_t off = 120 * (4 * qk + (lane >> 3)) + 16 * li;
      lo[k] = qk < full ? ld_nc8(p + off) : make_uint2(0u, 0u);
      hi[k] = qk < full && li < 7 ? ld_nc8(p + off + 8) : flag2;
    }
#pragma unroll
    for (int k = 0; k < kL128PackBatch; ++k) {
      const size_t qk = q + k * warps;
      if (qk < full)
        st_volatile(wire + 128 * (4 * qk + (lane >> 3)) + 16 * li, make_uint4(lo[k].x, lo[k].y, hi[k].x, hi[k].y));
    }
  }
  // the rest (the payload's last, partial quad, or all of an unaligned one)
  for (size_t q = full + (q0 + warps - full % warps) % warps; q < quads; q += warps) {
    const size_t j = 4 * q + (lane >> 3);
    if (j < lines) ll128_pack_slow(a, j, li);
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

// CTAs of `kernel` the GPU holds at once (cached per kernel)
template <class Kern>
static int resident_cap(Kern* kernel) {
  static int cap = 0;  // one per instantiation of this template, i.e. per kernel
  if (cap == 0) {
    int dev = 0, sms = 0, occ = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kLLThreads, 0);
    cap = (sms > 0 ? sms : 1) * (occ > 0 ? occ : 1);
  }
  return cap;
}

template <int DT, int NSRC>
static cudaError_t launch_ll_unpack_n(const LLArgs& a, int grid, cudaStream_t s) {
  auto* k = &ll_unpack_kernel<DT, NSRC>;
  const int cap = resident_cap(k);
  k<<<grid < cap ? grid : cap, kLLThreads, 0, s>>>(a);
  return cudaGetLastError();
}

template <int DT>
static cudaError_t ll_unpack_dt(const LLArgs& a, int grid, cudaStream_t s) {
  switch (a.nsrc) {
    case 1: return launch_ll_unpack_n<DT, 1>(a, grid, s);
    case 2: return launch_ll_unpack_n<DT, 2>(a, grid, s);
    case 3: return launch_ll_unpack_n<DT, 3>(a, grid, s);
    case 4: return launch_ll_unpack_n<DT, 4>(a, grid, s);
    case 5: return launch_ll_unpack_n<DT, 5>(a, grid, s);
    case 6: return launch_ll_unpack_n<DT, 6>(a, grid, s);
    case 7: return launch_ll_unpack_n<DT, 7>(a, grid, s);
    case 8: return launch_ll_unpack_n<DT, 8>(a, grid, s);
    default: return cudaErrorInvalidValue;
  }
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

RRA_UNPACK_DISPATCH(ll128_unpack_kernel)

cudaError_t launch_ll_unpack(int dt, const LLArgs& a, int grid, cudaStream_t s) {
  if (dt == RRA_INT32) return ll_unpack_dt<RRA_INT32>(a, grid, s);
  if (dt == RRA_FLOAT32) return ll_unpack_dt<RRA_FLOAT32>(a, grid, s);
  return ll_unpack_dt<RRA_BFLOAT16>(a, grid, s);
}

cudaError_t launch_ll128_unpack(int dt, const LLArgs& a, int grid, cudaStream_t s) {
  if (dt == RRA_INT32) return ll128_unpack_kernel_dt<RRA_INT32>(a, grid, s);
  if (dt == RRA_FLOAT32) return ll128_unpack_kernel_dt<RRA_FLOAT32>(a, grid, s);
  return ll128_unpack_kernel_dt<RRA_BFLOAT16>(a, grid, s);
}

}  // namespace rra
