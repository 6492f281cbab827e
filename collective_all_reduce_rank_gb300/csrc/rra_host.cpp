// rra_host.cpp -- the C ABI of include/rra.h: argument validation, the
// chunk plan, algorithm selection, launch planning, device status, the
// flight recorder and the tuning table.  Every computation of the
// collectives runs in the kernels (kernels_*.cu); this file only decides
// what to launch.
#include <cuda_runtime.h>
#include <dlfcn.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "rra.h"
#include "rra_internal.h"

using namespace rra;

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kDefaultWorkspace = 256ull << 20;
constexpr uint64_t kDefaultTimeoutNs = 500ull * 1000 * 1000;

struct DevState {
  bool ready = false;
  int sms = 0;
  char* base = nullptr;
  size_t bytes = 0;
  Workspace ws{};
};

DevState g_dev[kMaxDevices];
std::mutex g_dev_mu;
std::atomic<uint64_t> g_timeout_ns{0};
std::atomic<int> g_skip_rank{-1};
std::atomic<int> g_max_ctas{-1};  // -1: not set, read RRA_MAX_CTAS

// ---------------------------------------------------------------------------
// environment
// ---------------------------------------------------------------------------
long env_long(const char* name, long dflt) {
  const char* v = std::getenv(name);
  if (!v || !*v) return dflt;
  char* end = nullptr;
  const long x = std::strtol(v, &end, 10);
  return (end && *end == 0) ? x : dflt;
}

bool debug_on() {
  static const bool on = env_long("RRA_DEBUG", 0) != 0;
  return on;
}

uint64_t timeout_ns() {
  const uint64_t t = g_timeout_ns.load();
  if (t) return t;
  static const uint64_t env = (uint64_t)env_long("RRA_TIMEOUT_NS", 0);
  return env ? env : kDefaultTimeoutNs;
}

// Channels per rank the SM budget leaves a persistent kernel.
long channel_cap(int n) {
  const int m = rra::max_ctas_cap();
  return m > 0 ? std::max(1, m / n) : (long)kMaxChannels;
}

size_t elem_size(rra_dtype_t dt) { return dt == RRA_BFLOAT16 ? 2 : 4; }

const char* dtype_name(int dt) {
  return dt == RRA_INT32 ? "int32" : dt == RRA_FLOAT32 ? "float32" : dt == RRA_BFLOAT16 ? "bfloat16" : "?";
}

const char* algo_name(int a) {
  switch (a) {
    case RRA_ALGO_AUTO: return "auto";
    case RRA_ALGO_RING: return "ring";
    case RRA_ALGO_ONE_SHOT: return "one_shot";
    case RRA_ALGO_TWO_SHOT: return "two_shot";
    case RRA_ALGO_DIRECT: return "direct";
    case RRA_ALGO_COPY_ENGINE: return "copy_engine";
    case RRA_ALGO_TREE: return "tree";
    default: return "?";
  }
}

int parse_algo(const char* s) {
  if (!s) return -1;
  if (!std::strcmp(s, "ring")) return RRA_ALGO_RING;
  if (!std::strcmp(s, "one_shot") || !std::strcmp(s, "oneshot")) return RRA_ALGO_ONE_SHOT;
  if (!std::strcmp(s, "two_shot") || !std::strcmp(s, "twoshot")) return RRA_ALGO_TWO_SHOT;
  if (!std::strcmp(s, "direct")) return RRA_ALGO_DIRECT;
  if (!std::strcmp(s, "tree")) return RRA_ALGO_TREE;
  return -1;
}

// ---------------------------------------------------------------------------
// flight recorder: the last kRecent calls
// ---------------------------------------------------------------------------
constexpr int kRecent = 64;
struct CallRec {
  uint64_t seq;
  const char* call;
  int algo, n, dt, grid;
  size_t count;
  int status;
};
CallRec g_rec[kRecent];
uint64_t g_seq = 0;
std::mutex g_rec_mu;

rra_status_t record(const char* call, int algo, int n, size_t count, int dt, int grid,
                    rra_status_t st) {
  {
    std::lock_guard<std::mutex> lk(g_rec_mu);
    CallRec& c = g_rec[g_seq % kRecent];
    c = CallRec{g_seq, call, algo, n, dt, grid, count, (int)st};
    ++g_seq;
  }
  if (debug_on())
    std::fprintf(stderr, "[rra] %s algo=%s n=%d count=%zu dtype=%s grid=%d -> %s\n", call,
                 algo_name(algo), n, count, dtype_name(dt), grid, rra_status_string(st));
  return st;
}

// ---------------------------------------------------------------------------
// tuning table
// ---------------------------------------------------------------------------
struct TuneEntry {
  int n, dt, log2b, algo;
};
// The alpha-beta prior fitted on the box (per type and schedule): a call
// of S bytes per rank over n ranks takes alpha * syncs(n) + beta * n * S.
struct PriorEntry {
  int dt, algo;
  double alpha_us, beta_us_per_mib;
};
std::vector<TuneEntry> g_tune;
std::vector<PriorEntry> g_prior;
std::mutex g_tune_mu;

// Synchronizations of a schedule (the alpha count of the pages' model):
// 2(n-1) ring steps, one for one-shot, two for two-shot, 2 ceil(log2 n)
// for a tree.
double sync_steps(int algo, int n) {
  switch (algo) {
    case RRA_ALGO_RING: return 2.0 * (n - 1);
    case RRA_ALGO_ONE_SHOT: return 1.0;
    case RRA_ALGO_TWO_SHOT: return 2.0;
    case RRA_ALGO_TREE: {
      int l = 0;
      while ((1 << l) < n) ++l;
      return 2.0 * std::max(1, l);
    }
    default: return 1e30;
  }
}

int ceil_log2(size_t x) {
  int l = 0;
  while (((size_t)1 << l) < x && l < 63) ++l;
  return l;
}

// ---------------------------------------------------------------------------
// validation helpers
// ---------------------------------------------------------------------------
bool valid_dtype(int dt) { return dt == RRA_INT32 || dt == RRA_FLOAT32 || dt == RRA_BFLOAT16; }

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

bool overlap(const void* a, size_t an, const void* b, size_t bn) {
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return an && bn && x < y + bn && y < x + an;
}

// Input ranges may overlap one another (they are only read).  Output ranges
// must be pairwise disjoint, and an output may meet an input only as the
// exact in-place location allowed for that rank (inplace_in[r]).
rra_status_t check_alias(const void* const* in, size_t in_bytes, void* const* out, size_t out_bytes,
                         int n, const char* const* inplace_in) {
  for (int i = 0; i < n; ++i)
    for (int j = i + 1; j < n; ++j)
      if (overlap(out[i], out_bytes, out[j], out_bytes)) return RRA_ERR_ALIAS;
  for (int j = 0; j < n; ++j)
    for (int i = 0; i < n; ++i) {
      if (!overlap(out[j], out_bytes, in[i], in_bytes)) continue;
      if (i == j && inplace_in && in[i] == (const void*)inplace_in[i]) continue;
      return RRA_ERR_ALIAS;
    }
  return RRA_SUCCESS;
}

DevState* current_state(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  if (dev_out) *dev_out = dev;
  return &g_dev[dev];
}

int sm_count() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < kMaxDevices && g_dev[dev].ready) return g_dev[dev].sms;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

WaitCfg wait_cfg(DevState* s) {
  WaitCfg w;
  w.status = s->ws.status;
  w.sync = s->ws.sync;
  w.timeout_ns = timeout_ns();
  w.skip_rank = g_skip_rank.load();
  return w;
}

rra_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return RRA_SUCCESS;
  if (debug_on()) std::fprintf(stderr, "[rra] CUDA error: %s\n", cudaGetErrorString(e));
  return RRA_ERR_CUDA;
}

// Grid that gives every thread one unit (capped far above any real size;
// the kernels loop past it).
int cover_grid(size_t units, int threads) {
  const size_t want = (units + threads - 1) / threads;
  return (int)std::max<size_t>(1, std::min<size_t>(want, (size_t)1 << 30));
}

// Grid for a grid-stride streaming kernel: enough CTAs to give every
// thread work, at most what the GPU holds at once.
int stream_grid(size_t units, int threads, int per_sm) {
  const size_t want = (units + threads - 1) / threads;
  const size_t cap = (size_t)sm_count() * (size_t)per_sm;
  return (int)std::max<size_t>(1, std::min(want, cap));
}

// ---------------------------------------------------------------------------
// launch planning for the persistent kernels
// ---------------------------------------------------------------------------

rra_status_t run_twoshot(DevState* s, const void* const* in, void* const* out, int n, size_t count,
                         rra_dtype_t dt, bool vec, cudaStream_t st, int* grid_out) {
  TwoShotArgs a{};
  const size_t e = elem_size(dt), pu = 16 / e;
  const size_t per = (count + n - 1) / n;
  const size_t clen = (per + pu - 1) / pu * pu;
  for (int c = 0; c < n; ++c) {
    a.in[c] = in[c];
    a.out[c] = out[c];
    const size_t lo = std::min(count, (size_t)c * clen), hi = std::min(count, (size_t)(c + 1) * clen);
    a.chunk_lo[c] = lo;
    a.chunk_len[c] = hi - lo;
  }
  a.wait = wait_cfg(s);
  // Cluster form (TMA staging, exchange through distributed shared memory)
  // for aligned buffers; not with fault injection, whose silent rank would
  // leave its cluster peers at a hardware barrier.
  if (vec && n >= 2 && a.wait.skip_rank < 0 && env_long("RRA_TWOSHOT_CLUSTER", 0) != 0) {
    const int maxc = twoshot_cluster_max_clusters(n, dt);
    if (maxc > 0) {
      const size_t tu = (size_t)twoshot_cluster_tile_bytes(n) / 16;
      const size_t units0 = a.chunk_len[0] / pu;
      long c = std::min<long>({(long)maxc, (long)std::max<size_t>(1, (units0 + tu - 1) / tu), channel_cap(n)});
      c = std::min(c, env_long("RRA_TWOSHOT_CHANNELS", c));
      a.channels = (int)std::max(1L, c);
      *grid_out = n * a.channels;
      cudaError_t err = launch_twoshot_cluster(n, dt, a, n * a.channels, st);
      // the sub-unit tail of the last chunk (fewer than 16 bytes): same
      // ascending sum by the one-shot kernel
      size_t tail_lo = count;
      for (int c2 = 0; c2 < n; ++c2)
        if (a.chunk_len[c2] % pu) tail_lo = a.chunk_lo[c2] + a.chunk_len[c2] / pu * pu;
      if (err == cudaSuccess && tail_lo < count) {
        DirectArgs t{};
        for (int r = 0; r < n; ++r) {
          t.in[r] = static_cast<const char*>(in[r]) + tail_lo * e;
          t.out[r] = static_cast<char*>(out[r]) + tail_lo * e;
        }
        t.count = count - tail_lo;
        int g2 = 0;
        err = launch_oneshot(n, dt, false, t, 1, &g2, st);
      }
      return cuda_status(err);
    }
  }
  a.tile_units = twoshot_tile_units(n);
  a.lag = (int)std::max(0L, std::min(256L, env_long("RRA_TWOSHOT_LAG", 0)));
  int occ = 0;
  cudaError_t err = twoshot_occupancy(n, dt, vec, &occ);
  if (err != cudaSuccess || occ < 1) return cuda_status(err == cudaSuccess ? cudaErrorInvalidConfiguration : err);
  const size_t units0 = (a.chunk_len[0] + pu - 1) / pu;
  const size_t need = (units0 + a.tile_units - 1) / a.tile_units;
  // enough channels to fill every SM at the kernel's CTAs per SM, within the
  // progress words (one per rank, channel and warp) and the SM budget
  const long words_cap = (long)(kLinkFlags / ((size_t)n * kMaxWarps));
  const long budget_cap = rra::max_ctas_cap() > 0 ? channel_cap(n) : words_cap;
  long c = std::min<long>({words_cap, (long)(s->sms * occ / n), (long)std::max<size_t>(1, need), budget_cap});
  c = std::min(c, env_long("RRA_TWOSHOT_CHANNELS", c));
  if (c < 1) return RRA_ERR_UNSUPPORTED;
  a.channels = (int)c;
  a.progress = s->ws.flags + 2 * kLinkFlags;
  a.wait = wait_cfg(s);
  *grid_out = n * (int)c;
  return cuda_status(launch_twoshot(n, dt, vec, a, n * (int)c, st));
}

// The ring's form, by measured size ([AIH] "Protocols": LL for small
// messages, Simple for large ones).  RRA_RING_PROTO=ll | simple | staged
// forces one.  On 16-byte aligned buffers the staged form (Simple links,
// whole-CTA messages) is the fastest for large chunks; the per-warp LL form
// for small and mid-size ones, where both are bound by the ring's 2(n-1)
// hops and an LL hop is the cheaper.  Measured on GB300 (CUDA graph of 50
// calls, microseconds per call, LL against staged): fp32 at 8 ranks 15.6
// against 36.3 at 1 KiB per rank, 18.2 against 44.3 at 1 MiB, 41.3 against
// 46.7 at 2 MiB, then 72.3 against 50.7 at 4 MiB; at 4 ranks 8.5 against
// 16.3 at 1 KiB, 15.6 against 20.8 at 1 MiB, 31.3 against 22.0 at 2 MiB;
// at 2 ranks 4.9 against 6.4 at 1 KiB, 6.6 against 8.5 at 256 KiB, 8.8
// against 8.6 at 512 KiB.  bf16, whose LL lines carry fp32 partials: at 8
// ranks 30.7 against 45.5 at 1 MiB, 57.4 against 48.8 at 2 MiB; at 4 ranks
// 15.1 against 20.0 at 512 KiB, 23.1 against 21.1 at 1 MiB; at 2 ranks 8.1
// against 8.4 at 256 KiB, 11.1 against 8.5 at 512 KiB.  So LL takes chunks
// up to 256 KiB at n >= 3 and 128 KiB at n = 2, bf16 up to 128 KiB;
// RRA_RING_LL_STAGED_MAX_BYTES overrides the limit.  Without 16-byte
// alignment the per-warp LL form takes chunks up to RRA_RING_LL_MAX_BYTES
// (64 KiB) and the per-warp Simple form larger ones.
enum RingForm { kFormWarpSimple = 0, kFormWarpLL = 1, kFormStaged = 2 };

int ring_form(size_t chunk_bytes, bool staged_ok, int n, rra_dtype_t dt) {
  const char* p = std::getenv("RRA_RING_PROTO");
  if (p && !std::strcmp(p, "simple")) return kFormWarpSimple;
  if (p && !std::strcmp(p, "ll")) return kFormWarpLL;
  if (p && !std::strcmp(p, "staged") && staged_ok) return kFormStaged;
  if (staged_ok) {
    static const long ll_max = env_long("RRA_RING_LL_STAGED_MAX_BYTES", -1);
    const long lim = ll_max >= 0 ? ll_max
                     : dt == RRA_BFLOAT16 ? 128L << 10 : (n >= 3 ? 256L << 10 : 128L << 10);
    return (n >= 2 && (long)chunk_bytes <= lim) ? kFormWarpLL : kFormStaged;
  }
  static const long limit = env_long("RRA_RING_LL_MAX_BYTES", 64L << 10);
  return (long)chunk_bytes <= limit ? kFormWarpLL : kFormWarpSimple;
}

// Dynamic shared memory for the stages of the staged ring and tree
// (RRA_STAGED_SMEM_KB, 224 KB; a CTA may have 227 KB): at 224 KB a bfloat16
// ring tile of 1536 units (its partials travel as float32) still gets three
// stages, which it does not at 200.
static size_t staged_smem_budget() {
  static const size_t b = (size_t)std::max(16L, std::min(224L, env_long("RRA_STAGED_SMEM_KB", 224))) << 10;
  return b;
}

// Staged ring: messages of T units, G per step, K slots per link, D stages.
// Defaults (measured on GB300, 8 ranks x 100 MB per rank, T x G x K sweep):
// G = 6; T up to 2368 units for 4-byte types and up to 1536 for bfloat16
// (whose partials travel as float32), the largest tiles that still leave
// three stages (T 2304 with three stages: 0.347 ms; T 1728 with four:
// 0.364; T 2592 with two: 0.45); K = G + 3 (K = 2G keeps 1.3x the FIFO
// slots in L2 and measured 2-3% slower, K = G + 1 stalls on credits).
// Larger G fills L2 with FIFO slots (links x K x slot bytes) and runs
// slower.  Channels: as many as the GPU holds, but no more than
// leave G tiles of 128 units each; then T is the smallest multiple of 32
// units that covers the chunk in whole iterations, so no iteration runs
// nearly empty.  K drops to G + 1 when the FIFO would not fit the workspace.
rra_status_t run_ring_staged(DevState* s, RingArgs& a, size_t maxu, rra_dtype_t dt, cudaStream_t st,
                             int* grid_out) {
  const int n = a.n;
  const size_t aw = dt == RRA_BFLOAT16 ? 2 : 1;
  const long tmax = std::max(64L, std::min(4096L, env_long("RRA_RING_TILE", aw == 2 ? 1536 : 2368)));
  // G, messages per step, by the units u each channel carries of a chunk,
  // as measured best on GB300 (n = 4 and 8, fp32 and bf16, 128 KiB .. 16 MiB
  // per rank, G = 1 .. 8: every pick within 2% of the best): one message per
  // step while a step's message is small (u < 600), so no hop waits on
  // several; then 2 and 3, which let the next rank start on a step's first
  // messages; from 2600 units 4, as long as four messages cover the chunk in
  // one iteration, else 6 (more iterations: the messages of a step hide the
  // hop).  The old rule (up to 6 whenever 6 tiles of 128 units filled a
  // channel) was 10-35% slower from 1 to 16 MiB per rank.
  {
    const size_t ch_est = std::max<size_t>(1, (size_t)s->sms / n);
    const size_t u = (maxu + ch_est - 1) / ch_est;
    long g = 6;
    if (u < 600) g = 1;
    else if (u < 1300) g = 2;
    else if (u < 2600) g = 3;
    else if (u <= 4 * (size_t)tmax) g = 4;
    a.G = (int)std::max(1L, env_long("RRA_RING_G", g));
  }
  auto stages_for = [&](long t) {
    const long d = (long)(staged_smem_budget() / ((size_t)t * 16 * (1 + aw)));
    return (int)std::max(1L, std::min<long>({8L, d, env_long("RRA_RING_STAGES", 8)}));
  };
  int occ = 0;
  cudaError_t err = ring_staged_occupancy(dt, (int)tmax, stages_for(tmax), &occ);
  if (err != cudaSuccess || occ < 1) return cuda_status(err == cudaSuccess ? cudaErrorInvalidConfiguration : err);
  const long cmax = std::min<long>({(long)kMaxChannels, (long)(s->sms * occ / n), channel_cap(n)});
  if (cmax < 1) return RRA_ERR_UNSUPPORTED;
  const size_t G = (size_t)a.G;
  long c = std::min<long>({cmax, (long)std::max<size_t>(1, (maxu + G * 128 - 1) / (G * 128)),
                           env_long("RRA_RING_CHANNELS", cmax)});
  c = std::max(1L, c);
  const size_t iters = std::max<size_t>(1, (maxu + (size_t)c * G * tmax - 1) / ((size_t)c * G * tmax));
  long T = (long)((maxu + (size_t)c * G * iters - 1) / ((size_t)c * G * iters));
  T = std::max(32L, std::min(tmax, (T + 31) / 32 * 32));
  a.slice_units = (int)T;
  a.stages = stages_for(T);
  err = ring_staged_occupancy(dt, (int)T, a.stages, &occ);
  if (err != cudaSuccess || occ < 1) return cuda_status(err == cudaSuccess ? cudaErrorInvalidConfiguration : err);
  a.slot_bytes = (size_t)T * 16 * aw;
  a.K = (int)std::max((long)a.G + 1, env_long("RRA_RING_K", (long)a.G + 3));
  if ((size_t)c * n * a.K * a.slot_bytes > s->ws.fifo_bytes) a.K = a.G + 1;
  c = std::min<long>(c, (long)(s->ws.fifo_bytes / ((size_t)n * a.K * a.slot_bytes)));
  if (c < 1) return RRA_ERR_WORKSPACE;
  // messages per CTA stay below 2^31 (32-bit counters in the kernel)
  const size_t trips = (maxu + (size_t)c * a.G * T - 1) / ((size_t)c * a.G * T);
  if (trips * (size_t)(2 * n) * a.G >= (1ull << 31)) return RRA_ERR_UNSUPPORTED;
  a.channels = (int)c;
  a.fifo = s->ws.fifo;
  a.head = s->ws.flags;
  a.tail = s->ws.flags + kLinkFlags;
  *grid_out = n * (int)c;
  return cuda_status(launch_ring_staged(dt, a, n * (int)c, st));
}

// Staged double binary tree: the message split in two by the chunk plan for
// two parts (the first part on tree 0, the rest on tree 1); one message per
// tile of T units (T <= RRA_TREE_TILE: 2048 for 4-byte types, 1280 for
// bfloat16, whose partials travel as float32), G tiles per iteration
// (RRA_TREE_G; at most 24, 12 for bfloat16), K = G + 1 FIFO slots per up
// link (RRA_TREE_K), the broadcast L = 6 iterations behind the reduction
// (RRA_TREE_LAG), stages as shared memory allows; T balanced over whole
// iterations of one part as in the staged ring.  The limits are the best of
// a sweep on GB300 at 8 ranks x 100 MB (fp32: T 2048, G 12-24, L 6 within
// 1%; bfloat16: T 1280, G 12, L 6 0.663 ms against 0.700 for T 1024, G 24,
// L 4).
rra_status_t run_tree_staged(DevState* s, const void* const* in, void* const* out, int n, size_t count,
                             rra_dtype_t dt, cudaStream_t st, int* grid_out) {
  StagedTreeArgs a{};
  const size_t e = elem_size(dt), aw = dt == RRA_BFLOAT16 ? 2 : 1, pu = 16 / e;
  for (int r = 0; r < n; ++r) {
    a.in[r] = in[r];
    a.out[r] = out[r];
  }
  a.n = n;
  a.count = count;
  const size_t units = (count * e + 15) / 16;
  // chunk plan for two parts: H = ceil(count / 2) rounded up to whole units
  const size_t h = std::min(count, ((count + 1) / 2 + pu - 1) / pu * pu);
  a.half_units = (h + pu - 1) / pu;
  const size_t part = std::max(a.half_units, units - a.half_units);  // units of the larger part
  // G tiles per iteration (24 for the bucket), but no more than the part
  // fills with tiles of 128 units per channel: every message of a role
  // costs a synchronization even when it carries nothing, and a small
  // message is one up-and-back wave
  {
    const size_t ch_est = std::max<size_t>(1, (size_t)s->sms / n);
    const size_t fill = (part + ch_est * 128 - 1) / (ch_est * 128);
    const size_t gmax = aw == 2 ? 12 : 24;
    a.G = (int)std::max(1L, env_long("RRA_TREE_G", (long)std::max<size_t>(1, std::min(gmax, fill))));
  }
  a.lag = (int)std::max(1L, std::min(64L, env_long("RRA_TREE_LAG", 6)));
  const long tmax = std::max(64L, std::min(4096L, env_long("RRA_TREE_TILE", aw == 2 ? 1280 : 2048)));
  auto stages_for = [&](long t) {
    const long d = (long)(staged_smem_budget() / ((size_t)t * 16 * (1 + 2 * aw)));
    return (int)std::max(1L, std::min<long>({8L, d, env_long("RRA_TREE_STAGES", 8)}));
  };
  int occ = 0;
  cudaError_t err = tree_staged_occupancy(dt, (int)tmax, stages_for(tmax), &occ);
  if (err != cudaSuccess || occ < 1) return cuda_status(err == cudaSuccess ? cudaErrorInvalidConfiguration : err);
  const long cmax = std::min<long>({(long)kMaxChannels, (long)(s->sms * occ / n), channel_cap(n)});
  if (cmax < 1) return RRA_ERR_UNSUPPORTED;
  const size_t G = (size_t)a.G;
  long c = std::min<long>({cmax, (long)std::max<size_t>(1, (part + G * 128 - 1) / (G * 128)),
                           env_long("RRA_TREE_CHANNELS", cmax)});
  c = std::max(1L, c);
  const size_t iters = std::max<size_t>(1, (part + (size_t)c * G * tmax - 1) / ((size_t)c * G * tmax));
  long T = (long)((part + (size_t)c * G * iters - 1) / ((size_t)c * G * iters));
  T = std::max(32L, std::min(tmax, (T + 31) / 32 * 32));
  a.slice_units = (int)T;
  a.stages = stages_for(T);
  err = tree_staged_occupancy(dt, (int)T, a.stages, &occ);
  if (err != cudaSuccess || occ < 1) return cuda_status(err == cudaSuccess ? cudaErrorInvalidConfiguration : err);
  a.slot_bytes = (size_t)T * 16 * aw;
  a.K = (int)std::max((long)a.G + 1, env_long("RRA_TREE_K", (long)a.G + 1));
  // one up FIFO per rank and channel (a rank sends up in one tree at most;
  // the totals come down from outputs)
  if ((size_t)c * n * a.K * a.slot_bytes > s->ws.fifo_bytes) a.K = a.G + 1;
  c = std::min<long>(c, (long)(s->ws.fifo_bytes / ((size_t)n * a.K * a.slot_bytes)));
  if (c < 1 || (size_t)2 * n * c > kLinkFlags) return RRA_ERR_WORKSPACE;
  // messages per CTA (both trees) stay below 2^31
  const size_t trips = (part + (size_t)c * a.G * T - 1) / ((size_t)c * a.G * T);
  if (trips * 4 * (size_t)a.G >= (1ull << 31)) return RRA_ERR_UNSUPPORTED;
  a.channels = (int)c;
  a.fifo = s->ws.fifo;
  a.head = s->ws.flags;
  a.tail = s->ws.flags + kLinkFlags;
  a.joined = s->ws.flags + 2 * kLinkFlags;  // the two-shot progress words, unused by a tree call
  a.wait = wait_cfg(s);
  *grid_out = n * (int)c;
  return cuda_status(launch_tree_staged(dt, a, n * (int)c, st));
}

// LL double tree (small messages): warp tiles of 32 x kTreeLLUnits units,
// one per warp while the SMs hold enough CTAs of 8 warps (more tiles loop);
// both line regions of every rank (up: units x AW x 32 bytes, down: units x
// 32) must fit the workspace's LL region.
rra_status_t run_tree_ll(DevState* s, const void* const* in, void* const* out, int n, size_t count,
                         rra_dtype_t dt, cudaStream_t st, int* grid_out) {
  TreeLLArgs a{};
  const size_t e = elem_size(dt), aw = dt == RRA_BFLOAT16 ? 2 : 1, pu = 16 / e;
  for (int r = 0; r < n; ++r) {
    a.in[r] = in[r];
    a.out[r] = out[r];
  }
  a.n = n;
  a.count = count;
  const size_t units = (count * e + 15) / 16;
  // chunk plan for two parts, as the staged tree
  const size_t h = std::min(count, ((count + 1) / 2 + pu - 1) / pu * pu);
  a.half_units = (h + pu - 1) / pu;
  a.up_bytes = units * aw * 32;
  a.dn_bytes = units * 32;
  if ((size_t)n * (a.up_bytes + a.dn_bytes) > s->ws.ll_bytes) return RRA_ERR_WORKSPACE;
  const size_t part = std::max(a.half_units, units - a.half_units);
  const size_t tu = 32 * (size_t)kTreeLLUnits, warps = kTreeLLThreads / 32;
  const size_t tiles = (part + tu - 1) / tu;
  int occ = 0;
  cudaError_t err = tree_ll_occupancy(dt, &occ);
  if (err != cudaSuccess || occ < 1) return cuda_status(err == cudaSuccess ? cudaErrorInvalidConfiguration : err);
  long c = std::min<long>({(long)std::max<size_t>(1, (tiles + warps - 1) / warps), (long)(s->sms * occ / n),
                           channel_cap(n), env_long("RRA_TREE_CHANNELS", kMaxChannels)});
  if (c < 1) return RRA_ERR_UNSUPPORTED;
  a.channels = (int)c;
  a.lines = s->ws.ll;
  a.joined = s->ws.flags + 2 * kLinkFlags;  // the two-shot progress words, unused by a tree call
  a.wait = wait_cfg(s);
  *grid_out = n * (int)c;
  return cuda_status(launch_tree_ll(dt, a, n * (int)c, st));
}

// The tree's form: RRA_TREE_PROTO=ll | staged forces one; by default LL
// lines for messages up to tree_ll_max_bytes per rank whose lines fit the
// LL region, the staged tree above.  Measured on GB300 (CUDA graph of 50
// calls, microseconds per call, LL against staged): fp32 at 8 ranks 7.4
// against 20.6 at 1 KiB per rank, 9.3 against 26.7 at 256 KiB, 11.6
// against 30.7 at 512 KiB; at 2 ranks 4.3 against 8.1 at 1 KiB, 10.2
// against 13.3 at 2 MiB; bf16 at 8 ranks 8.3 against 20.6 at 1 KiB, 22.0
// against 30.9 at 512 KiB; at 2 ranks 9.5 against 11.3 at 1 MiB and 15.1
// against 13.5 at 2 MiB; with the 64 MiB region, up to the largest
// messages whose lines fit, fp32 at 2 ranks x 8 MiB 26.8 against 32.8, at
// 4 x 4 MiB 26.4 against 48.2, at 8 x 2 MiB 24.1 against 55.8, bf16 at 4
// ranks x 2 MiB 30.6 against 29.5 (within the run-to-run spread).  So LL
// wherever its lines fit, but for bf16 at 2 ranks above 1 MiB per rank.
size_t tree_ll_max_bytes(int n, rra_dtype_t dt);

rra_status_t run_tree(DevState* s, const void* const* in, void* const* out, int n, size_t count, rra_dtype_t dt,
                      cudaStream_t st, int* grid_out) {
  const char* p = std::getenv("RRA_TREE_PROTO");
  if (p && !std::strcmp(p, "ll")) return run_tree_ll(s, in, out, n, count, dt, st, grid_out);
  if (p && !std::strcmp(p, "staged")) return run_tree_staged(s, in, out, n, count, dt, st, grid_out);
  const size_t e = elem_size(dt), aw = dt == RRA_BFLOAT16 ? 2 : 1;
  const size_t units = (count * e + 15) / 16;
  if (count * e <= tree_ll_max_bytes(n, dt) && (size_t)n * units * 32 * (aw + 1) <= s->ws.ll_bytes)
    return run_tree_ll(s, in, out, n, count, dt, st, grid_out);
  return run_tree_staged(s, in, out, n, count, dt, st, grid_out);
}

size_t tree_ll_max_bytes(int n, rra_dtype_t dt) {
  static const long lim = env_long("RRA_TREE_LL_MAX_BYTES", -1);
  if (lim >= 0) return (size_t)lim;
  return dt == RRA_BFLOAT16 && n == 2 ? (size_t)1 << 20 : SIZE_MAX;
}

// mode: kRingAllReduce / kRingReduceScatter / kRingAllGather.  ibase, obase,
// len: per chunk, in elements.
rra_status_t run_ring(DevState* s, const void* const* in, void* const* out, int n, int mode,
                      const size_t* ibase, const size_t* obase, const size_t* len, rra_dtype_t dt,
                      bool vec, cudaStream_t st, int* grid_out) {
  RingArgs a{};
  const size_t e = elem_size(dt), pu = 16 / e;
  size_t maxu = 0;
  for (int c = 0; c < n; ++c) {
    a.in[c] = in[c];
    a.out[c] = out[c];
    a.ibase[c] = ibase[c];
    a.obase[c] = obase[c];
    a.len[c] = len[c];
    maxu = std::max(maxu, (len[c] + pu - 1) / pu);
  }
  a.n = n;
  a.mode = mode;
  a.wait = wait_cfg(s);
  // Cluster form: the ring's links in distributed shared memory, tiles by
  // bulk copies.  It needs 16-byte aligned buffers and chunk starts, whole
  // units in every chunk but the last, and no fault injection (a silent
  // rank would leave its cluster at a hardware barrier).
  bool cluster_ok = vec && n >= 2 && a.wait.skip_rank < 0 && env_long("RRA_RING_CLUSTER", 0) != 0;
  for (int c = 0; c < n && cluster_ok; ++c) {
    cluster_ok = (ibase[c] * e) % 16 == 0 && (obase[c] * e) % 16 == 0;
    if (c + 1 < n && len[c] % pu) cluster_ok = cluster_ok && mode == kRingAllReduce && len[c + 1] == 0;
  }
  if (cluster_ok && mode != kRingAllReduce)
    for (int c = 0; c < n; ++c) cluster_ok = cluster_ok && len[c] % pu == 0;
  const int maxc = cluster_ok ? ring_cluster_max_clusters(n, dt) : 0;
  if (maxc > 0) {
    a.G = (int)std::max(1L, std::min((long)ring_cluster_slots(dt) / 2, env_long("RRA_RING_G", ring_cluster_slots(dt) / 2)));
    a.K = ring_cluster_slots(dt);
    const size_t tu = (size_t)ring_cluster_tile_units(dt);
    size_t wmax = 0;
    for (int c = 0; c < n; ++c) wmax = std::max(wmax, len[c] / pu);
    const size_t need = (wmax + (size_t)a.G * tu - 1) / ((size_t)a.G * tu);
    long c = std::min<long>({(long)maxc, (long)std::max<size_t>(1, need), channel_cap(n)});
    c = std::min(c, env_long("RRA_RING_CHANNELS", c));
    a.channels = (int)std::max(1L, c);
    *grid_out = n * a.channels;
    cudaError_t err = launch_ring_cluster(dt, a, n * a.channels, st);
    // sub-unit tail of the ragged chunk: the ring's order for that chunk,
    // x_{c+1}, ..., x_{c-1}, x_c, by the one-shot kernel on rotated inputs
    for (int c = 0; c < n && err == cudaSuccess; ++c) {
      if (len[c] % pu == 0) continue;
      const size_t done = len[c] / pu * pu;
      DirectArgs t{};
      for (int k = 0; k < n; ++k) {
        const int src = (c + 1 + k) % n;
        t.in[k] = static_cast<const char*>(in[src]) + (ibase[c] + done) * e;
        t.out[k] = static_cast<char*>(out[k]) + (obase[c] + done) * e;
      }
      t.count = len[c] - done;
      int g2 = 0;
      err = launch_oneshot(n, dt, false, t, 1, &g2, st);
    }
    return cuda_status(err);
  }
  bool staged_ok = vec;
  for (int c = 0; c < n; ++c) staged_ok = staged_ok && (ibase[c] * e) % 16 == 0 && (obase[c] * e) % 16 == 0;
  const int form = ring_form(maxu * 16, staged_ok, n, dt);
  if (form == kFormStaged) return run_ring_staged(s, a, maxu, dt, st, grid_out);
  const int proto = form == kFormWarpLL ? kProtoLL : kProtoSimple;
  a.slice_units = kRingThreads * ring_units_per_thread(dt, proto);
  // Credits: a rank's sends minus receives never exceed G.  Simple raises a
  // credit per message, so K > G keeps n full FIFOs from all being pending
  // at once (with K == G every rank could fill its FIFO in the first step
  // and wait for a credit its successor gives only after sending too).  LL
  // raises one credit per G messages, which lags by up to G-1 more, so it
  // needs K >= 2G.
  // G: 4, or fewer when 16 channels of G messages would be mostly empty
  const size_t gfill = (maxu + 16 * (size_t)a.slice_units - 1) / (16 * (size_t)a.slice_units);
  a.G = (int)std::max(1L, env_long("RRA_RING_G", std::min<long>(4, (long)std::max<size_t>(1, gfill))));
  // LL: at least 16 slots, so a small message's 2(n-1) steps rarely wait
  // for a credit (measured 35 us against 44 at 8 ranks x 1 KiB)
  const long kmin = proto == kProtoLL ? 2L * a.G : (long)a.G + 1;
  a.K = (int)std::max(kmin, env_long("RRA_RING_K", proto == kProtoLL ? std::max(2L * a.G, 16L) : 2L * a.G));
  const int aw = dt == RRA_BFLOAT16 ? 2 : 1;
  a.slot_bytes = (size_t)a.slice_units * aw * (proto == kProtoLL ? 32 : 16);
  int occ = 0;
  cudaError_t err = ring_occupancy(dt, vec, proto, &occ);
  if (err != cudaSuccess || occ < 1) return cuda_status(err == cudaSuccess ? cudaErrorInvalidConfiguration : err);
  const size_t need = (maxu + (size_t)a.G * a.slice_units - 1) / ((size_t)a.G * a.slice_units);
  // LL lines live in their own region (never a raw word under a poll)
  const size_t fifo_cap = (proto == kProtoLL ? s->ws.ll_bytes : s->ws.fifo_bytes) / ((size_t)n * a.K * a.slot_bytes);
  long c = std::min<long>({(long)kMaxChannels, (long)(s->sms * occ / n), (long)std::max<size_t>(1, need),
                           (long)fifo_cap, env_long("RRA_RING_CHANNELS", 16), channel_cap(n)});
  if (fifo_cap < 1) {
    // a small workspace's LL region may not hold one channel of LL slots;
    // the staged form sizes its slots by the message (unless a form was
    // forced)
    if (proto == kProtoLL && staged_ok && !std::getenv("RRA_RING_PROTO"))
      return run_ring_staged(s, a, maxu, dt, st, grid_out);
    return RRA_ERR_WORKSPACE;
  }
  if (c < 1) return RRA_ERR_UNSUPPORTED;
  if (proto == kProtoLL) {
    // LL line flags carry the slot round in 12 bits: more rounds than that
    // in one call go over the Simple protocol instead
    const size_t iters = (maxu + (size_t)c * a.G * a.slice_units - 1) / ((size_t)c * a.G * a.slice_units);
    const size_t sends = mode == kRingAllReduce ? 2 * (size_t)(n - 1) : (size_t)(n - 1);
    if (iters * sends * a.G / a.K >= 4096) {
      a.slice_units = kRingThreads * ring_units_per_thread(dt, kProtoSimple);
      a.K = (int)std::max((long)a.G + 1, env_long("RRA_RING_K", 2L * a.G));
      a.slot_bytes = (size_t)a.slice_units * aw * 16;
      err = ring_occupancy(dt, vec, kProtoSimple, &occ);
      if (err != cudaSuccess || occ < 1) return cuda_status(err == cudaSuccess ? cudaErrorInvalidConfiguration : err);
      const size_t cap2 = s->ws.fifo_bytes / ((size_t)n * a.K * a.slot_bytes);
      c = std::min<long>({(long)kMaxChannels, (long)(s->sms * occ / n), (long)std::max<size_t>(1, need),
                          (long)cap2, env_long("RRA_RING_CHANNELS", 16), channel_cap(n)});
      if (cap2 < 1) return RRA_ERR_WORKSPACE;
      if (c < 1) return RRA_ERR_UNSUPPORTED;
      a.channels = (int)c;
      a.fifo = s->ws.fifo;
      a.head = s->ws.flags;
      a.tail = s->ws.flags + kLinkFlags;
      *grid_out = n * (int)c;
      return cuda_status(launch_ring(dt, vec, kProtoSimple, a, n * (int)c, st));
    }
  }
  a.channels = (int)c;
  a.fifo = proto == kProtoLL ? s->ws.ll : s->ws.fifo;
  a.head = s->ws.flags;
  a.tail = s->ws.flags + kLinkFlags;
  a.wait = wait_cfg(s);
  if (proto == kProtoLL) {
    // messages per link in this call; with no more than K, no slot is
    // reused and no sender waits for a credit
    const size_t iters = (maxu + (size_t)c * a.G * a.slice_units - 1) / ((size_t)c * a.G * a.slice_units);
    const size_t sends = mode == kRingAllReduce ? 2 * (size_t)(n - 1) : (size_t)(n - 1);
    a.no_credits = iters * sends * (size_t)a.G <= (size_t)a.K ? 1 : 0;
  }
  *grid_out = n * (int)c;
  return cuda_status(launch_ring(dt, vec, proto, a, n * (int)c, st));
}

bool all_aligned16(const void* const* p, int n) {
  for (int i = 0; i < n; ++i)
    if (!aligned(p[i], 16)) return false;
  return true;
}

// The measured table shipped beside the library (tune/gb300.txt next to
// librra.so), or RRA_TUNING_FILE; loaded once, on the first rra_init.
void load_default_tuning() {
  static std::once_flag once;
  std::call_once(once, [] {
    const char* env = std::getenv("RRA_TUNING_FILE");
    if (env && *env) {
      rra_load_tuning(env);
      return;
    }
    Dl_info info;
    if (!dladdr(reinterpret_cast<void*>(&rra_load_tuning), &info) || !info.dli_fname) return;
    std::string path(info.dli_fname);
    const size_t slash = path.rfind('/');
    path = (slash == std::string::npos ? std::string(".") : path.substr(0, slash)) + "/tune/gb300.txt";
    if (FILE* f = std::fopen(path.c_str(), "r")) {
      std::fclose(f);
      rra_load_tuning(path.c_str());
    }
  });
}

}  // namespace

uint64_t rra::current_timeout_ns() { return timeout_ns(); }

int rra::current_skip_rank() { return g_skip_rank.load(); }

long rra::channels_allowed(int n) { return channel_cap(n); }

rra_status_t rra::record_call(const char* call, int algo, int n, size_t count, int dt, int grid, rra_status_t st) {
  return record(call, algo, n, count, dt, grid, st);
}

// Prefer the wait on a peer that never posted: it names the rank that did
// not join, not one stuck behind it.
void rra::decode_status(const DevStatus& h, int32_t info[4]) {
  const unsigned long long d = h.root_detail ? h.root_detail : h.detail;
  const int peer = (int)((d >> 16) & 0xFFFF);
  info[0] = h.code;
  info[1] = (int)(d & 0xFFFF);
  info[2] = peer == 0xFFFF ? -1 : peer;
  info[3] = (int)((d >> 32) & 0x7FFFFFFF);
}

int rra::max_ctas_cap() {
  int m = g_max_ctas.load();
  if (m < 0) {
    static const int env = (int)env_long("RRA_MAX_CTAS", 0);
    m = env > 0 ? env : 0;
  }
  return m;
}

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" {

const char* rra_status_string(rra_status_t s) {
  switch (s) {
    case RRA_SUCCESS: return "success";
    case RRA_ERR_INVALID_ARG: return "invalid argument";
    case RRA_ERR_UNSUPPORTED: return "unsupported";
    case RRA_ERR_ALIAS: return "buffers overlap";
    case RRA_ERR_NOT_INITIALIZED: return "rra_init was not called for this device";
    case RRA_ERR_CUDA: return "CUDA error";
    case RRA_ERR_TIMEOUT: return "device wait timed out";
    case RRA_ERR_WORKSPACE: return "workspace too small for the call (rra_init workspace_bytes)";
    default: return "unknown status";
  }
}

rra_status_t rra_init(int device, size_t workspace_bytes) {
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev || device >= kMaxDevices)
    return RRA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (cudaSetDevice(device) != cudaSuccess) return RRA_ERR_CUDA;
  DevState& s = g_dev[device];
  if (s.ready) return RRA_SUCCESS;
  size_t bytes = workspace_bytes ? workspace_bytes : kDefaultWorkspace;
  bytes = std::max<size_t>(bytes, 1u << 20);
  char* p = nullptr;
  if (cudaMalloc(&p, bytes) != cudaSuccess) return RRA_ERR_CUDA;
  if (cudaMemset(p, 0, bytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    cudaFree(p);
    return RRA_ERR_CUDA;
  }
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  s.base = p;
  s.bytes = bytes;
  s.sms = sms;
  s.ws.status = reinterpret_cast<DevStatus*>(p);
  s.ws.sync = reinterpret_cast<SyncHdr*>(p + 64);
  s.ws.flags = reinterpret_cast<uint64_t*>(p + kFlagOffset);
  s.ws.fifo = p + kFifoOffset;
  const size_t slots = bytes > kFifoOffset ? (bytes - kFifoOffset) / 256 * 256 : 0;
  // LL lines: 64 MiB (the per-warp LL ring's 16 channels x 16 slots of
  // 32 KiB per link at 8 ranks x 256 KiB chunks; the LL tree's lines up to
  // 1 MiB per rank at 8 ranks), at most half the slot space
  s.ws.ll_bytes = std::min<size_t>(64ull << 20, slots / 2 / 256 * 256);
  s.ws.fifo_bytes = slots - s.ws.ll_bytes;
  s.ws.ll = s.ws.fifo + s.ws.fifo_bytes;
  s.ready = true;
  load_default_tuning();
  return RRA_SUCCESS;
}

rra_status_t rra_finalize(void) {
  std::lock_guard<std::mutex> lk(g_dev_mu);
  int cur = 0;
  const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
  rra_status_t st = RRA_SUCCESS;
  for (int d = 0; d < kMaxDevices; ++d) {
    DevState& s = g_dev[d];
    if (!s.ready) continue;
    if (cudaSetDevice(d) != cudaSuccess || cudaFree(s.base) != cudaSuccess) st = RRA_ERR_CUDA;
    s = DevState{};
  }
  if (have_cur) cudaSetDevice(cur);
  return st;
}

void rra_set_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns); }

void rra_set_max_ctas(int max_ctas) { g_max_ctas.store(max_ctas < 0 ? 0 : max_ctas); }

void rra_debug_skip_rank(int rank) { g_skip_rank.store(rank); }

rra_algo_t rra_select_algo(int nranks, size_t bytes_per_rank, rra_dtype_t dtype) {
  if (nranks <= 1) return RRA_ALGO_ONE_SHOT;
  std::lock_guard<std::mutex> lk(g_tune_mu);
  {
    const int lb = ceil_log2(std::max<size_t>(1, bytes_per_rank));
    int best_l = -1, best_a = -1;
    for (const TuneEntry& t : g_tune)
      if (t.n == nranks && t.dt == (int)dtype && t.log2b <= lb && t.log2b > best_l) {
        best_l = t.log2b;
        best_a = t.algo;
      }
    if (best_a >= 0) return (rra_algo_t)best_a;
  }
  // Prior: the alpha-beta model of the "Algorithms" section with alpha and
  // beta fitted on this GPU (the "ab" lines of the tuning table): the
  // schedule with the least alpha * syncs(n) + beta * n * S.
  double best_t = 0;
  int best = -1;
  const double nS_mib = (double)nranks * (double)bytes_per_rank / (1024.0 * 1024.0);
  for (const PriorEntry& p : g_prior) {
    if (p.dt != (int)dtype) continue;
    const double t = p.alpha_us * sync_steps(p.algo, nranks) + p.beta_us_per_mib * nS_mib;
    if (best < 0 || t < best_t) {
      best_t = t;
      best = p.algo;
    }
  }
  if (best >= 0) return (rra_algo_t)best;
  // No measurement at all (no table loaded): the same model with one GPU's
  // traffic, where the n ranks' peer reads of a unit are the same HBM bytes,
  // so every schedule moves 2nS and one-shot has the fewest syncs.
  return RRA_ALGO_ONE_SHOT;
}

rra_status_t rra_load_tuning(const char* path) {
  if (!path) {
    std::lock_guard<std::mutex> lk(g_tune_mu);
    g_tune.clear();
    g_prior.clear();
    return RRA_SUCCESS;
  }
  FILE* f = std::fopen(path, "r");
  if (!f) return RRA_ERR_INVALID_ARG;
  std::vector<TuneEntry> t;
  std::vector<PriorEntry> pr;
  char line[256];
  bool bad = false;
  while (std::fgets(line, sizeof line, f)) {
    char* hash = std::strchr(line, '#');
    if (hash) *hash = 0;
    char dts[32], al[32];
    int n = 0, lb = 0;
    double alpha = 0, beta = 0;
    if (std::sscanf(line, " ab %31s %31s %lf %lf", dts, al, &alpha, &beta) == 4) {
      const int dt = !std::strcmp(dts, "int32") ? RRA_INT32 : !std::strcmp(dts, "float32") ? RRA_FLOAT32
                     : !std::strcmp(dts, "bfloat16") ? RRA_BFLOAT16 : -1;
      const int a = parse_algo(al);
      if (dt < 0 || a < 0 || a == RRA_ALGO_DIRECT || !(alpha >= 0) || !(beta > 0)) {
        bad = true;
        break;
      }
      pr.push_back(PriorEntry{dt, a, alpha, beta});
      continue;
    }
    const int got = std::sscanf(line, "%d %31s %d %31s", &n, dts, &lb, al);
    if (got <= 0) continue;
    if (got != 4) { bad = true; break; }
    int dt = !std::strcmp(dts, "int32") ? RRA_INT32 : !std::strcmp(dts, "float32") ? RRA_FLOAT32
             : !std::strcmp(dts, "bfloat16") ? RRA_BFLOAT16 : -1;
    const int a = parse_algo(al);
    if (dt < 0 || a < 0 || a == RRA_ALGO_DIRECT || n < 1 || n > kMaxRanks || lb < 0 || lb > 63) {
      bad = true;
      break;
    }
    t.push_back(TuneEntry{n, dt, lb, a});
  }
  std::fclose(f);
  if (bad) return RRA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_tune_mu);
  g_tune.swap(t);
  g_prior.swap(pr);
  return RRA_SUCCESS;
}

rra_status_t rra_allreduce(const void* const* bufs, void* const* outs, int nranks, size_t count,
                           rra_dtype_t dtype, rra_op_t op, rra_algo_t algo, rra_stream_t stream) {
  const char* call = "allreduce";
  if (!bufs || !outs || nranks < 1 || !valid_dtype(dtype) || op != RRA_SUM || (int)algo < 0 ||
      ((int)algo > RRA_ALGO_TWO_SHOT && algo != RRA_ALGO_TREE))
    return record(call, algo, nranks, count, dtype, 0,
                  nranks > kMaxRanks ? RRA_ERR_UNSUPPORTED : RRA_ERR_INVALID_ARG);
  if (nranks > kMaxRanks) return record(call, algo, nranks, count, dtype, 0, RRA_ERR_UNSUPPORTED);
  const size_t e = elem_size(dtype);
  if (count > (SIZE_MAX / 2) / e) return record(call, algo, nranks, count, dtype, 0, RRA_ERR_INVALID_ARG);
  if (algo == RRA_ALGO_TREE && nranks > 1) {
    for (int r = 0; r < nranks; ++r)
      if (!bufs[r] || !outs[r] || !aligned(bufs[r], 16) || !aligned(outs[r], 16))
        return record(call, algo, nranks, count, dtype, 0, RRA_ERR_UNSUPPORTED);
  }
  for (int r = 0; r < nranks; ++r)
    if (!bufs[r] || !outs[r] || !aligned(bufs[r], e) || !aligned(outs[r], e))
      return record(call, algo, nranks, count, dtype, 0, RRA_ERR_INVALID_ARG);
  const size_t S = count * e;
  const rra_status_t al = check_alias(bufs, S, outs, S, nranks, reinterpret_cast<const char* const*>(outs));
  if (al != RRA_SUCCESS) return record(call, algo, nranks, count, dtype, 0, al);
  if (algo == RRA_ALGO_AUTO) {
    const int env = parse_algo(std::getenv("RRA_ALGO"));
    algo = (env == RRA_ALGO_RING || env == RRA_ALGO_ONE_SHOT || env == RRA_ALGO_TWO_SHOT ||
            (env == RRA_ALGO_TREE && all_aligned16(bufs, nranks) && all_aligned16((const void* const*)outs, nranks)))
               ? (rra_algo_t)env
               : rra_select_algo(nranks, S, dtype);
    // the tree moves 16-byte units by bulk copies: other buffers take
    // one-shot, the schedule with the fewest syncs
    if (algo == RRA_ALGO_TREE && !(all_aligned16(bufs, nranks) && all_aligned16((const void* const*)outs, nranks)))
      algo = RRA_ALGO_ONE_SHOT;
  }
  if (count == 0) return record(call, algo, nranks, count, dtype, 0, RRA_SUCCESS);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool vec = all_aligned16(bufs, nranks) && all_aligned16((const void* const*)outs, nranks);
  bool inplace_all = true;
  for (int r = 0; r < nranks; ++r) inplace_all = inplace_all && bufs[r] == outs[r];
  if (nranks == 1) {
    if (inplace_all) return record(call, algo, 1, count, dtype, 0, RRA_SUCCESS);
    DirectArgs a{};
    a.in[0] = bufs[0];
    a.out[0] = outs[0];
    a.count = count;
    int grid = 0;
    const cudaError_t err = launch_oneshot(1, dtype, vec, a, (count * e + 15) / 16, &grid, st);
    return record(call, algo, 1, count, dtype, grid, cuda_status(err));
  }
  if (algo == RRA_ALGO_ONE_SHOT) {
    DirectArgs a{};
    for (int r = 0; r < nranks; ++r) {
      a.in[r] = bufs[r];
      a.out[r] = outs[r];
    }
    a.count = count;
    // the literal per-rank form reads every input while other ranks write
    // their outputs, so in place it would need the barrier one-shot has
    // between its reads and writes on n GPUs; in place takes the combined
    // form, which reads a unit of all n inputs before it writes any output
    a.per_rank_grid = (int)env_long("RRA_ONESHOT_PER_RANK", 0) != 0 && !inplace_all;
    if (vec && !a.per_rank_grid && env_long("RRA_ONESHOT_TMA", 0) != 0 && count * e >= 16) {
      // whole 16-byte units by bulk copies, the sub-unit tail by the LSU kernel
      const size_t units = count * e / 16;
      DevState* s = current_state(nullptr);
      DevStatus* status = (s && s->ready) ? s->ws.status : nullptr;
      int grid = 0;
      cudaError_t err = launch_oneshot_tma(nranks, dtype, bufs, outs, units, status, timeout_ns(), &grid, st);
      const size_t done = units * 16 / e;
      if (err == cudaSuccess && done < count) {
        DirectArgs t{};
        for (int r = 0; r < nranks; ++r) {
          t.in[r] = static_cast<const char*>(bufs[r]) + done * e;
          t.out[r] = static_cast<char*>(outs[r]) + done * e;
        }
        t.count = count - done;
        int g2 = 0;
        err = launch_oneshot(nranks, dtype, false, t, 1, &g2, st);
      }
      return record(call, algo, nranks, count, dtype, grid, cuda_status(err));
    }
    int grid = 0;
    const cudaError_t err = launch_oneshot(nranks, dtype, vec, a, (count * e + 15) / 16, &grid, st);
    return record(call, algo, nranks, count, dtype, grid, cuda_status(err));
  }
  int dev = 0;
  DevState* s = current_state(&dev);
  if (!s || !s->ready) return record(call, algo, nranks, count, dtype, 0, RRA_ERR_NOT_INITIALIZED);
  int grid = 0;
  rra_status_t rs;
  if (algo == RRA_ALGO_TREE) {
    rs = run_tree(s, bufs, outs, nranks, count, dtype, st, &grid);
  } else if (algo == RRA_ALGO_TWO_SHOT) {
    rs = run_twoshot(s, bufs, outs, nranks, count, dtype, vec, st, &grid);
  } else {
    const size_t pu = 16 / e;
    const size_t per = (count + nranks - 1) / nranks;
    const size_t clen = (per + pu - 1) / pu * pu;
    size_t lo[kMaxRanks], len[kMaxRanks];
    for (int c = 0; c < nranks; ++c) {
      lo[c] = std::min(count, (size_t)c * clen);
      len[c] = std::min(count, (size_t)(c + 1) * clen) - lo[c];
    }
    rs = run_ring(s, bufs, outs, nranks, kRingAllReduce, lo, lo, len, dtype, vec, st, &grid);
  }
  return record(call, algo, nranks, count, dtype, grid, rs);
}

rra_status_t rra_reduce_scatter(const void* const* bufs, void* const* outs, int nranks,
                                size_t recvcount, rra_dtype_t dtype, rra_op_t op, rra_algo_t algo,
                                rra_stream_t stream) {
  const char* call = "reduce_scatter";
  if (!bufs || !outs || nranks < 1 || !valid_dtype(dtype) || op != RRA_SUM || (int)algo < 0 ||
      (int)algo > RRA_ALGO_DIRECT || algo == RRA_ALGO_ONE_SHOT)
    return record(call, algo, nranks, recvcount, dtype, 0,
                  nranks > kMaxRanks ? RRA_ERR_UNSUPPORTED : RRA_ERR_INVALID_ARG);
  if (nranks > kMaxRanks) return record(call, algo, nranks, recvcount, dtype, 0, RRA_ERR_UNSUPPORTED);
  const size_t e = elem_size(dtype);
  if (recvcount > (SIZE_MAX / 2) / e / kMaxRanks)
    return record(call, algo, nranks, recvcount, dtype, 0, RRA_ERR_INVALID_ARG);
  for (int r = 0; r < nranks; ++r)
    if (!bufs[r] || !outs[r] || !aligned(bufs[r], e) || !aligned(outs[r], e))
      return record(call, algo, nranks, recvcount, dtype, 0, RRA_ERR_INVALID_ARG);
  const size_t rbytes = recvcount * e;
  const char* inplace[kMaxRanks];
  for (int r = 0; r < nranks; ++r) inplace[r] = static_cast<const char*>(bufs[r]) + (size_t)r * rbytes;
  // an in-place output sits inside its own input: allowed only at slice r
  for (int r = 0; r < nranks; ++r)
    if (overlap(outs[r], rbytes, bufs[r], rbytes * nranks) && (const char*)outs[r] != inplace[r])
      return record(call, algo, nranks, recvcount, dtype, 0, RRA_ERR_ALIAS);
  {
    const void* ins[kMaxRanks];
    for (int r = 0; r < nranks; ++r) ins[r] = bufs[r];
    // outputs pairwise disjoint, and no output inside another rank's input
    for (int i = 0; i < nranks; ++i)
      for (int j = 0; j < nranks; ++j) {
        if (i != j && overlap(outs[i], rbytes, outs[j], rbytes))
          return record(call, algo, nranks, recvcount, dtype, 0, RRA_ERR_ALIAS);
        if (i != j && overlap(outs[j], rbytes, ins[i], rbytes * nranks))
          return record(call, algo, nranks, recvcount, dtype, 0, RRA_ERR_ALIAS);
      }
  }
  if (algo == RRA_ALGO_AUTO) algo = RRA_ALGO_DIRECT;
  if (algo == RRA_ALGO_TWO_SHOT) algo = RRA_ALGO_DIRECT;
  if (recvcount == 0) return record(call, algo, nranks, recvcount, dtype, 0, RRA_SUCCESS);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool vec = all_aligned16(bufs, nranks) && all_aligned16((const void* const*)outs, nranks) &&
                   (rbytes % 16) == 0;
  if (algo == RRA_ALGO_DIRECT || nranks == 1) {
    DirectArgs a{};
    for (int r = 0; r < nranks; ++r) {
      a.in[r] = bufs[r];
      a.out[r] = outs[r];
    }
    a.count = recvcount;
    int grid = 0;
    const cudaError_t err = launch_direct_rs(nranks, dtype, vec, a, (rbytes + 15) / 16, &grid, st);
    return record(call, algo, nranks, recvcount, dtype, grid, cuda_status(err));
  }
  DevState* s = current_state(nullptr);
  if (!s || !s->ready) return record(call, algo, nranks, recvcount, dtype, 0, RRA_ERR_NOT_INITIALIZED);
  size_t ib[kMaxRanks], ob[kMaxRanks], len[kMaxRanks];
  for (int c = 0; c < nranks; ++c) {
    ib[c] = (size_t)c * recvcount;
    ob[c] = 0;
    len[c] = recvcount;
  }
  int grid = 0;
  const rra_status_t rs =
      run_ring(s, bufs, outs, nranks, kRingReduceScatter, ib, ob, len, dtype, vec, st, &grid);
  return record(call, algo, nranks, recvcount, dtype, grid, rs);
}

rra_status_t rra_all_gather(const void* const* bufs, void* const* outs, int nranks, size_t sendcount,
                            rra_dtype_t dtype, rra_algo_t algo, rra_stream_t stream) {
  const char* call = "all_gather";
  if (!bufs || !outs || nranks < 1 || !valid_dtype(dtype) || (int)algo < 0 ||
      (int)algo > RRA_ALGO_COPY_ENGINE || algo == RRA_ALGO_ONE_SHOT)
    return record(call, algo, nranks, sendcount, dtype, 0,
                  nranks > kMaxRanks ? RRA_ERR_UNSUPPORTED : RRA_ERR_INVALID_ARG);
  if (nranks > kMaxRanks) return record(call, algo, nranks, sendcount, dtype, 0, RRA_ERR_UNSUPPORTED);
  const size_t e = elem_size(dtype);
  if (sendcount > (SIZE_MAX / 2) / e / kMaxRanks)
    return record(call, algo, nranks, sendcount, dtype, 0, RRA_ERR_INVALID_ARG);
  for (int r = 0; r < nranks; ++r)
    if (!bufs[r] || !outs[r] || !aligned(bufs[r], e) || !aligned(outs[r], e))
      return record(call, algo, nranks, sendcount, dtype, 0, RRA_ERR_INVALID_ARG);
  const size_t sbytes = sendcount * e;
  for (int i = 0; i < nranks; ++i)
    for (int j = 0; j < nranks; ++j) {
      if (i != j && overlap(outs[i], sbytes * nranks, outs[j], sbytes * nranks))
        return record(call, algo, nranks, sendcount, dtype, 0, RRA_ERR_ALIAS);
      if (!overlap(outs[j], sbytes * nranks, bufs[i], sbytes)) continue;
      // in place: shard i sits at slot i of its own output
      if (i == j && bufs[i] == static_cast<const char*>(outs[i]) + (size_t)i * sbytes) continue;
      return record(call, algo, nranks, sendcount, dtype, 0, RRA_ERR_ALIAS);
    }
  if (algo == RRA_ALGO_AUTO || algo == RRA_ALGO_TWO_SHOT) algo = RRA_ALGO_DIRECT;
  if (sendcount == 0) return record(call, algo, nranks, sendcount, dtype, 0, RRA_SUCCESS);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (algo == RRA_ALGO_COPY_ENGINE) {
    // one device-to-device copy per (destination, shard); the shard already
    // in place is skipped
    cudaError_t err = cudaSuccess;
    for (int r = 0; r < nranks && err == cudaSuccess; ++r)
      for (int q = 0; q < nranks && err == cudaSuccess; ++q) {
        char* dst = static_cast<char*>(outs[r]) + (size_t)q * sbytes;
        if (dst == bufs[q]) continue;
        err = cudaMemcpyAsync(dst, bufs[q], sbytes, cudaMemcpyDeviceToDevice, st);
      }
    return record(call, algo, nranks, sendcount, dtype, 0, cuda_status(err));
  }
  const bool vec = all_aligned16(bufs, nranks) && all_aligned16((const void* const*)outs, nranks) &&
                   (sbytes % 16) == 0;
  if (algo == RRA_ALGO_DIRECT || nranks == 1) {
    DirectArgs a{};
    for (int r = 0; r < nranks; ++r) {
      a.in[r] = bufs[r];
      a.out[r] = outs[r];
    }
    a.count = sendcount;
    int grid = 0;
    const cudaError_t err = launch_direct_ag(nranks, dtype, vec, a, (sbytes + 15) / 16, &grid, st);
    return record(call, algo, nranks, sendcount, dtype, grid, cuda_status(err));
  }
  DevState* s = current_state(nullptr);
  if (!s || !s->ready) return record(call, algo, nranks, sendcount, dtype, 0, RRA_ERR_NOT_INITIALIZED);
  size_t ib[kMaxRanks], ob[kMaxRanks], len[kMaxRanks];
  for (int c = 0; c < nranks; ++c) {
    ib[c] = 0;
    ob[c] = (size_t)c * sendcount;
    len[c] = sendcount;
  }
  int grid = 0;
  const rra_status_t rs =
      run_ring(s, bufs, outs, nranks, kRingAllGather, ib, ob, len, dtype, vec, st, &grid);
  return record(call, algo, nranks, sendcount, dtype, grid, rs);
}

rra_status_t rra_allreduce_rmsnorm(const void* const* bufs, void* const* outs, int nranks,
                                   size_t rows, size_t hidden, const void* gamma, float eps,
                                   rra_dtype_t dtype, rra_stream_t stream) {
  const char* call = "allreduce_rmsnorm";
  const size_t count = rows * hidden;
  if (!bufs || !outs || !gamma || nranks < 1 || (dtype != RRA_FLOAT32 && dtype != RRA_BFLOAT16) ||
      hidden == 0 || !(eps >= 0.f))
    return record(call, RRA_ALGO_ONE_SHOT, nranks, count, dtype, 0,
                  nranks > kMaxRanks ? RRA_ERR_UNSUPPORTED : RRA_ERR_INVALID_ARG);
  if (nranks > kMaxRanks || hidden > kNormMaxHidden || rows > 0x7FFFFFFFull)
    return record(call, RRA_ALGO_ONE_SHOT, nranks, count, dtype, 0, RRA_ERR_UNSUPPORTED);
  const size_t e = elem_size(dtype);
  if (rows && hidden > (SIZE_MAX / 4) / rows / e)
    return record(call, RRA_ALGO_ONE_SHOT, nranks, count, dtype, 0, RRA_ERR_INVALID_ARG);
  if (!aligned(gamma, e)) return record(call, RRA_ALGO_ONE_SHOT, nranks, count, dtype, 0, RRA_ERR_INVALID_ARG);
  for (int r = 0; r < nranks; ++r)
    if (!bufs[r] || !outs[r] || !aligned(bufs[r], e) || !aligned(outs[r], e))
      return record(call, RRA_ALGO_ONE_SHOT, nranks, count, dtype, 0, RRA_ERR_INVALID_ARG);
  const size_t S = count * e;
  rra_status_t al = check_alias(bufs, S, outs, S, nranks, reinterpret_cast<const char* const*>(outs));
  for (int r = 0; r < nranks && al == RRA_SUCCESS; ++r)
    if (overlap(outs[r], S, gamma, hidden * e)) al = RRA_ERR_ALIAS;
  if (al != RRA_SUCCESS) return record(call, RRA_ALGO_ONE_SHOT, nranks, count, dtype, 0, al);
  if (rows == 0) return record(call, RRA_ALGO_ONE_SHOT, nranks, 0, dtype, 0, RRA_SUCCESS);
  const bool vec = all_aligned16(bufs, nranks) && all_aligned16((const void* const*)outs, nranks) &&
                   aligned(gamma, 16) && (hidden * e) % 16 == 0;
  const cudaError_t err = launch_allreduce_rmsnorm(nranks, dtype, vec, bufs, outs, gamma, rows, hidden, eps,
                                                   reinterpret_cast<cudaStream_t>(stream));
  return record(call, RRA_ALGO_ONE_SHOT, nranks, count, dtype, (int)rows, cuda_status(err));
}

size_t rra_ll_wire_bytes(size_t payload_bytes) { return 8 * ((payload_bytes + 3) / 4); }

size_t rra_ll128_wire_bytes(size_t payload_bytes) { return 128 * ((payload_bytes + 119) / 120); }

static rra_status_t pack_common(const char* call, bool is128, const void* payload,
                                size_t payload_bytes, void* wire, uint64_t flag, rra_stream_t stream) {
  if (!payload || !wire || flag == 0 || !aligned(wire, 16) || payload_bytes > (SIZE_MAX / 4))
    return record(call, 0, 1, payload_bytes, -1, 0, RRA_ERR_INVALID_ARG);
  const size_t wbytes = is128 ? rra_ll128_wire_bytes(payload_bytes) : rra_ll_wire_bytes(payload_bytes);
  if (overlap(payload, payload_bytes, wire, wbytes))
    return record(call, 0, 1, payload_bytes, -1, 0, RRA_ERR_ALIAS);
  if (payload_bytes == 0) return record(call, 0, 1, 0, -1, 0, RRA_SUCCESS);
  LLArgs a{};
  a.payload = payload;
  a.wire_out = wire;
  a.payload_bytes = payload_bytes;
  a.flag = flag;
  a.vec = aligned(payload, 16);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int grid;
  cudaError_t e;
  if (is128) {
    const size_t quads = (payload_bytes + 479) / 480;
    // From 64 MiB a grid that covers the payload in one trip of eight
    // quads a warp (the kernel's batch), so the block scheduler balances
    // the SMs; below, a resident grid-stride grid.  Measured on GB300
    // against the resident grid, four sources: 0.885 -> 0.947 of the HBM
    // copy rate at 256 MiB, 0.893 -> 0.998 at 1 GiB, equal at 16-64 MiB
    // (one quad a warp over a covering grid was slower than either).
    const size_t per_cta = (size_t)(kLLThreads / 32) * kL128PackBatch;
    grid = payload_bytes >= ((size_t)64 << 20) ? (int)std::max<size_t>(1, (quads + per_cta - 1) / per_cta)
                                                : stream_grid(quads * 32, kLLThreads, 8);
    e = launch_ll128_pack(a, grid, st);
  } else {
    grid = cover_grid((payload_bytes + 15) / 16, kLLThreads);
    e = launch_ll_pack(a, grid, st);
  }
  return record(call, 0, 1, payload_bytes, -1, grid, cuda_status(e));
}

static rra_status_t unpack_common(const char* call, bool is128, const void* const* wires, int nsrc,
                                  void* out, size_t payload_bytes, rra_dtype_t dtype, rra_op_t op,
                                  uint64_t expected, rra_stream_t stream) {
  if (!wires || !out || nsrc < 1 || !valid_dtype(dtype) || op != RRA_SUM || expected == 0 ||
      payload_bytes % elem_size(dtype) || !aligned(out, elem_size(dtype)) || payload_bytes > (SIZE_MAX / 4))
    return record(call, 0, nsrc, payload_bytes, dtype, 0,
                  nsrc > kMaxRanks ? RRA_ERR_UNSUPPORTED : RRA_ERR_INVALID_ARG);
  if (nsrc > kMaxRanks) return record(call, 0, nsrc, payload_bytes, dtype, 0, RRA_ERR_UNSUPPORTED);
  const size_t wbytes = is128 ? rra_ll128_wire_bytes(payload_bytes) : rra_ll_wire_bytes(payload_bytes);
  for (int k = 0; k < nsrc; ++k) {
    if (!wires[k] || !aligned(wires[k], 16)) return record(call, 0, nsrc, payload_bytes, dtype, 0, RRA_ERR_INVALID_ARG);
    if (overlap(wires[k], wbytes, out, payload_bytes))
      return record(call, 0, nsrc, payload_bytes, dtype, 0, RRA_ERR_ALIAS);
  }
  if (payload_bytes == 0) return record(call, 0, nsrc, 0, dtype, 0, RRA_SUCCESS);
  DevState* s = current_state(nullptr);
  if (!s || !s->ready) return record(call, 0, nsrc, payload_bytes, dtype, 0, RRA_ERR_NOT_INITIALIZED);
  LLArgs a{};
  for (int k = 0; k < nsrc; ++k) a.wire_in[k] = wires[k];
  a.out = out;
  a.payload_bytes = payload_bytes;
  a.flag = expected;
  a.nsrc = nsrc;
  a.vec = aligned(out, 16);
  a.wait = wait_cfg(s);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int grid;
  cudaError_t e;
  if (is128) {
    const size_t quads = (payload_bytes + 479) / 480;
    grid = stream_grid(quads * 32, kLLThreads, 8);
    e = launch_ll128_unpack(dtype, a, grid, st);
  } else {
    grid = stream_grid((payload_bytes + 15) / 16, kLLThreads, 8);
    e = launch_ll_unpack(dtype, a, grid, st);
  }
  return record(call, 0, nsrc, payload_bytes, dtype, grid, cuda_status(e));
}

rra_status_t rra_ll_pack(const void* payload, size_t payload_bytes, void* wire, uint32_t flag,
                         rra_stream_t stream) {
  return pack_common("ll_pack", false, payload, payload_bytes, wire, flag, stream);
}

rra_status_t rra_ll128_pack(const void* payload, size_t payload_bytes, void* wire, uint64_t flag,
                            rra_stream_t stream) {
  return pack_common("ll128_pack", true, payload, payload_bytes, wire, flag, stream);
}

rra_status_t rra_ll_unpack(const void* const* wires, int nsrc, void* out, size_t payload_bytes,
                           rra_dtype_t dtype, rra_op_t op, uint32_t expected_flag,
                           rra_stream_t stream) {
  return unpack_common("ll_unpack", false, wires, nsrc, out, payload_bytes, dtype, op, expected_flag,
                       stream);
}

rra_status_t rra_ll128_unpack(const void* const* wires, int nsrc, void* out, size_t payload_bytes,
                              rra_dtype_t dtype, rra_op_t op, uint64_t expected_flag,
                              rra_stream_t stream) {
  return unpack_common("ll128_unpack", true, wires, nsrc, out, payload_bytes, dtype, op,
                       expected_flag, stream);
}

rra_status_t rra_query_status(rra_stream_t stream, int32_t info[4]) {
  if (info) info[0] = info[1] = info[2] = info[3] = 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return RRA_ERR_CUDA;
  DevState* s = current_state(nullptr);
  if (!s || !s->ready) return RRA_SUCCESS;
  DevStatus h{};
  if (cudaMemcpy(&h, s->ws.status, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return RRA_ERR_CUDA;
  if (h.code == 0) return RRA_SUCCESS;
  if (info) decode_status(h, info);
  // clear the record; the abort tag belongs to a finished call and can stay
  DevStatus z{};
  z.abort_tag = h.abort_tag;
  if (cudaMemcpy(s->ws.status, &z, sizeof z, cudaMemcpyHostToDevice) != cudaSuccess) return RRA_ERR_CUDA;
  return (rra_status_t)h.code;
}

int rra_dump_recent(char* buf, size_t len) {
  std::lock_guard<std::mutex> lk(g_rec_mu);
  std::string s;
  const uint64_t first = g_seq > kRecent ? g_seq - kRecent : 0;
  int count = 0;
  for (uint64_t q = first; q < g_seq; ++q) {
    const CallRec& c = g_rec[q % kRecent];
    char line[256];
    std::snprintf(line, sizeof line, "%llu %s algo=%s n=%d count=%zu dtype=%s grid=%d status=%s\n",
                  (unsigned long long)c.seq, c.call, algo_name(c.algo), c.n, c.count,
                  dtype_name(c.dt), c.grid, rra_status_string((rra_status_t)c.status));
    s += line;
    ++count;
  }
  if (buf && len) {
    const size_t m = std::min(len - 1, s.size());
    std::memcpy(buf, s.data(), m);
    buf[m] = 0;
  }
  return count;
}

}  // extern "C"
