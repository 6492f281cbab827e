// rra_internal.h -- what the host runtime (rra_host.cpp) and the kernel
// files share: workspace layout, kernel argument structs, launchers.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "rra.h"

namespace rra {

constexpr int kMaxRanks = RRA_MAX_RANKS;
constexpr int kMaxChannels = 80;  // CTAs per virtual rank in persistent kernels (76 = 152 SMs / 2 ranks)

// ---------------------------------------------------------------------------
// workspace (one per device, made by rra_init, zero-filled)
//
//   [0, 64)        DevStatus: first device error + abort tag
//   [64, 128)      SyncHdr: call epoch + end-of-kernel arrival counter
//   [256, ...)     step flags, one uint64 per (link or rank, channel, warp):
//                  ring head, ring tail, two-shot progress
//   [kFifoOffset, +fifo_bytes) FIFO slots of raw data (the staged ring and
//                  tree, the per-warp Simple ring)
//   [ll, end)      LL lines (the per-warp LL ring, the LL tree), 64 MiB,
//                  at most half the slots: a region that only ever holds LL
//                  lines, so that a poll never meets a raw data word that
//                  happens to equal its flag
// ---------------------------------------------------------------------------
// A wait that expires records where: bit 63 set, bits 32..62 index (step
// or line), bits 16..31 the rank waited for (0xFFFF: none), bits 0..15 the
// waiting rank or LL source.  `detail` keeps the first such record;
// `root_detail` one whose awaited peer posted nothing at all in the call
// (the rank that never joined, rather than one stuck behind it).
struct DevStatus {
  int32_t code;                    // 0 or the first rra_status_t recorded on the device
  uint32_t abort_tag;              // == tag of the call that gave up (epoch + 1)
  unsigned long long detail;       // first expired wait
  unsigned long long root_detail;  // expired wait on a peer that never posted
  uint32_t pad[10];
};
static_assert(sizeof(DevStatus) == 64, "status block is one 64-byte line");

struct SyncHdr {
  uint32_t epoch;   // bumped by the last CTA of every synchronizing kernel
  uint32_t arrive;  // CTAs of the running kernel that have finished
  uint32_t pad[14];
};

constexpr int kMaxWarps = 16;  // warps per CTA of the persistent kernels (512 threads)
constexpr size_t kFlagOffset = 256;
constexpr size_t kLinkFlags = (size_t)kMaxRanks * kMaxChannels * kMaxWarps;
constexpr size_t kFlagWords = 3 * kLinkFlags;  // ring head | ring tail | two-shot progress
constexpr size_t kFifoOffset = 256 * 1024;
static_assert(kFlagOffset + kFlagWords * 8 <= kFifoOffset, "flags fit below the FIFO");

struct Workspace {
  DevStatus* status;
  SyncHdr* sync;
  uint64_t* flags;  // kFlagWords entries
  char* fifo;
  size_t fifo_bytes;
  char* ll;
  size_t ll_bytes;
};

// Settings every waiting kernel gets by value.
struct WaitCfg {
  DevStatus* status;
  SyncHdr* sync;
  uint64_t timeout_ns;
  int skip_rank;  // fault injection: this rank posts nothing (-1: off)
};

// ---------------------------------------------------------------------------
// kernel arguments
// ---------------------------------------------------------------------------

// One-shot all-reduce, direct reduce-scatter, direct all-gather.
struct DirectArgs {
  const void* in[kMaxRanks];
  void* out[kMaxRanks];
  size_t count;       // elements per unit range (AR: count, RS: recvcount, AG: sendcount)
  int per_rank_grid;  // one-shot: 1 -> gridDim.y = n, block row r writes only out[r]
};

// Two-shot all-reduce (fused, persistent, cooperative).
struct TwoShotArgs {
  const void* in[kMaxRanks];
  void* out[kMaxRanks];
  size_t chunk_lo[kMaxRanks];   // element offset of chunk c
  size_t chunk_len[kMaxRanks];  // elements in chunk c
  uint64_t* progress;           // [(rank * channels + ch) * warps + warp]
  int channels;
  int tile_units;  // 16-byte units per tile per iteration
  int lag;         // tiles the gather trails the reduce by (0: the measured default)
  WaitCfg wait;
};

// Ring (persistent, cooperative): all-reduce, reduce-scatter or all-gather,
// with the Simple or the LL protocol on its links.
enum RingMode : int { kRingAllReduce = 0, kRingReduceScatter = 1, kRingAllGather = 2 };
enum RingProto : int { kProtoSimple = 0, kProtoLL = 1 };

struct RingArgs {
  const void* in[kMaxRanks];
  void* out[kMaxRanks];
  size_t ibase[kMaxRanks];  // element offset of chunk c inside a rank's input
  size_t obase[kMaxRanks];  // element offset of chunk c inside a rank's output
  size_t len[kMaxRanks];    // elements in chunk c
  char* fifo;               // links * slots * slot_bytes
  uint64_t* head;           // [link * warps + warp]: messages posted by the sender
  uint64_t* tail;           // [link * warps + warp]: messages consumed by the receiver
  size_t slot_bytes;
  int n;
  int channels;
  int mode;
  int slice_units;  // 16-byte units per message (= blockDim * units per thread)
  int G;            // messages per step and iteration
  int K;            // FIFO slots per link
  int stages;       // staged form: shared-memory stages per CTA
  int no_credits;   // per-warp LL form: no slot is reused in this call, so
                    // receivers raise no credits (the sender never waits)
  WaitCfg wait;
};

// Staged double binary tree all-reduce (persistent, cooperative).  A rank
// sends up and posts down in at most one of the two trees, so per channel:
// up FIFO of rank r at link r; heads [2n x channels] (up, then down); tails
// [n x channels] (up); joined flags [n x channels].
struct StagedTreeArgs {
  const void* in[kMaxRanks];
  void* out[kMaxRanks];
  size_t count;       // elements per rank
  size_t half_units;  // 16-byte units of the part reduced on tree 0 (the rest: tree 1)
  char* fifo;    // n up links x channels x K slots x slot_bytes
  uint64_t* head;
  uint64_t* tail;
  uint64_t* joined;  // [n x channels]: the call's epoch once the CTA has started
  size_t slot_bytes;
  int n;
  int channels;
  int slice_units;  // 16-byte units per message
  int G;            // tiles per iteration
  int K;            // FIFO slots per link
  int stages;       // shared-memory stages per CTA
  int lag;          // iterations the broadcast trails the reduction by (>= 1)
  WaitCfg wait;
};

// LL double binary tree all-reduce for small messages (persistent,
// cooperative): every node posts its partial as LL lines in its up region,
// every node with children its totals in its down region; each line is
// written once per call, so no slot is reused and no credit is needed.
// Rank r's regions: up at lines + r * (up_bytes + dn_bytes) (unit u's
// accumulator words at u * AW * 32), down right after (unit u at u * 32).
struct TreeLLArgs {
  const void* in[kMaxRanks];
  void* out[kMaxRanks];
  size_t count;       // elements per rank
  size_t half_units;  // 16-byte units of the part reduced on tree 0 (the rest: tree 1)
  char* lines;
  size_t up_bytes;    // per rank: units x AW x 32
  size_t dn_bytes;    // per rank: units x 32
  uint64_t* joined;   // [n x channels]: the call's epoch once the CTA has started
  int n;
  int channels;
  WaitCfg wait;
};

struct LLArgs {
  const void* wire_in[kMaxRanks];
  void* out;
  const void* payload;
  void* wire_out;
  size_t payload_bytes;
  uint64_t flag;  // pack: flag to write; unpack: expected flag
  int nsrc;
  int vec;  // payload / out 16-byte aligned
  WaitCfg wait;
};

// ---------------------------------------------------------------------------
// launchers (kernels_*.cu); all return the launch's cudaError_t
// ---------------------------------------------------------------------------
constexpr int kDirectThreads = 512;
constexpr int kRingThreads = 512;
constexpr int kRingUnitsPerThread = 2;
// per-warp ring: units per lane per message.  LL takes one: a lane then
// polls 32 bytes of lines a word group (64 for bfloat16, whose partials are
// fp32) and keeps them in registers, where two units spilled (measured on
// GB300: 1.1-1.4x faster for fp32 and 1.2-1.8x for bfloat16 at 4-8 ranks x
// 1 KiB-1 MiB per rank).
#ifdef __CUDACC__
__host__ __device__
#endif
constexpr int ring_units_per_thread(int dt, int proto) { return proto == kProtoLL ? 1 : kRingUnitsPerThread; }
// Two-shot: 16-byte units per thread per tile, and the CTAs per SM its
// kernel is compiled for: two, so that twice the warps hide the loads'
// latency (on GB300, 2 ranks x 64-256 MiB fp32: one CTA per SM with 4
// units a lane reached 0.62-0.64 of the HBM copy rate, two 0.74-0.75).  Up
// to four ranks every warp reduces and gathers (64 registers a thread: 2
// units a lane at two ranks, 1 at three and four).  From five ranks a lane
// holding n inputs and n-1 sums would need the registers of one CTA per
// SM, so the kernel splits each CTA's warps into reducers (n inputs) and
// gatherers (n-1 sums), and a tile is then the reducers' units (8 ranks x
// 64-256 MiB: 0.81-0.82 fused, 0.86-0.90 split; up to four ranks the split
// measured 2-15% slower than the fused form).
#ifdef __CUDACC__
__host__ __device__
#endif
constexpr int twoshot_units_per_thread(int n) { return n >= 3 ? 1 : 2; }
#ifdef __CUDACC__
__host__ __device__
#endif
constexpr int twoshot_min_blocks(int n) { return 2; }
#ifdef __CUDACC__
__host__ __device__
#endif
constexpr bool twoshot_split(int n) { return n >= 5; }
#ifdef __CUDACC__
__host__ __device__
#endif
constexpr int twoshot_tile_units(int n) {
  return twoshot_split(n) ? kDirectThreads / 2 : kDirectThreads * twoshot_units_per_thread(n);
}
constexpr int kLLThreads = 256;
// LL128 pack: quads per warp per trip, every load in flight before the stores
constexpr int kL128PackBatch = 8;

// SM budget set by rra_set_max_ctas (0: none); kernels_direct.cu caps its
// grids with it.
int max_ctas_cap();

// Settings of rra_host.cpp that the allocation-free entry point
// (noalloc.cu) honours too: the bound of device waits
// (rra_set_timeout_ns), the rank fault injection silences
// (rra_debug_skip_rank), the channels per rank the SM budget leaves, the
// flight recorder, and the decoding of a status block into {code, rank,
// peer, index}.
uint64_t current_timeout_ns();
int current_skip_rank();
long channels_allowed(int n);
rra_status_t record_call(const char* call, int algo, int n, size_t count, int dt, int grid, rra_status_t st);
void decode_status(const DevStatus& h, int32_t info[4]);

// Streaming kernels: `units` 16-byte units per grid row; *grid receives the
// CTAs per row launched.
cudaError_t launch_oneshot(int n, int dt, bool vec, const DirectArgs& a, size_t units, int* grid,
                           cudaStream_t s);
cudaError_t launch_direct_rs(int n, int dt, bool vec, const DirectArgs& a, size_t units, int* grid,
                             cudaStream_t s);
cudaError_t launch_direct_ag(int n, int dt, bool vec, const DirectArgs& a, size_t units, int* grid,
                             cudaStream_t s);

// One-shot with bulk-copy staging: whole 16-byte units only, 16-byte
// aligned buffers; status may be null.
cudaError_t launch_oneshot_tma(int n, int dt, const void* const* in, void* const* out, size_t units,
                               DevStatus* status, uint64_t timeout_ns, int* grid, cudaStream_t s);

// All-reduce + RMSNorm, one CTA per row (hidden <= kNormMaxHidden).
constexpr size_t kNormMaxHidden = 51200;
cudaError_t launch_allreduce_rmsnorm(int n, int dt, bool vec, const void* const* in, void* const* out,
                                     const void* gamma, size_t rows, size_t hidden, float eps,
                                     cudaStream_t s);

// Persistent kernels are launched cooperatively: every CTA is resident or
// the launch fails.  *max_blocks_per_sm reports the occupancy limit.
cudaError_t twoshot_occupancy(int n, int dt, bool vec, int* max_blocks_per_sm);
cudaError_t launch_twoshot(int n, int dt, bool vec, const TwoShotArgs& a, int grid, cudaStream_t s);
// Two-shot on thread-block clusters of n CTAs (n in [2, 8]): whole 16-byte
// units, 16-byte aligned buffers; grid = n * clusters.
int twoshot_cluster_tile_bytes(int n);
int twoshot_cluster_max_clusters(int n, int dt);
cudaError_t launch_twoshot_cluster(int n, int dt, const TwoShotArgs& a, int grid, cudaStream_t s);

// Ring on thread-block clusters of n CTAs: whole 16-byte units, 16-byte
// aligned chunk starts; a.G tiles per step (< the compiled slot count).
int ring_cluster_tile_units(int dt);
int ring_cluster_slots(int dt);
int ring_cluster_max_clusters(int n, int dt);
cudaError_t launch_ring_cluster(int dt, const RingArgs& a, int grid, cudaStream_t s);

// Ring with whole-CTA messages staged in shared memory (Simple protocol):
// 16-byte aligned buffers and chunk starts; one link counter per (link,
// channel); a.slice_units units per message, a.stages stages.
size_t ring_staged_smem(int dt, int tile_units, int stages);
cudaError_t ring_staged_occupancy(int dt, int tile_units, int stages, int* max_blocks_per_sm);
cudaError_t launch_ring_staged(int dt, const RingArgs& a, int grid, cudaStream_t s);

// LL tree: 16-byte aligned buffers; kTreeLLThreads threads, each lane
// kTreeLLUnits units per tile.  One unit a lane: more warps share a message
// and fewer polled lines sit in each lane (measured on GB300 against two:
// 1.1-1.4x faster for fp32 and bfloat16 from 16 KiB to 256 KiB per rank at
// 2-8 ranks; 0.88-0.97x for bfloat16 at 8 ranks x 512 KiB-1 MiB and 2
// ranks x 1 MiB).
constexpr int kTreeLLThreads = 256;
constexpr int kTreeLLUnits = 1;
cudaError_t tree_ll_occupancy(int dt, int* max_blocks_per_sm);
cudaError_t launch_tree_ll(int dt, const TreeLLArgs& a, int grid, cudaStream_t s);

// Staged tree: 16-byte aligned buffers.
size_t tree_staged_smem(int dt, int tile_units, int stages);
cudaError_t tree_staged_occupancy(int dt, int tile_units, int stages, int* max_blocks_per_sm);
cudaError_t launch_tree_staged(int dt, const StagedTreeArgs& a, int grid, cudaStream_t s);

cudaError_t ring_occupancy(int dt, bool vec, int proto, int* max_blocks_per_sm);
cudaError_t launch_ring(int dt, bool vec, int proto, const RingArgs& a, int grid, cudaStream_t s);

cudaError_t launch_ll_pack(const LLArgs& a, int grid, cudaStream_t s);
cudaError_t launch_ll_unpack(int dt, const LLArgs& a, int grid, cudaStream_t s);
cudaError_t launch_ll128_pack(const LLArgs& a, int grid, cudaStream_t s);
cudaError_t launch_ll128_unpack(int dt, const LLArgs& a, int grid, cudaStream_t s);

}  // namespace rra
