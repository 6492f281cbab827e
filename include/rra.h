/*
 * rra.h -- all-reduce, reduce-scatter and all-gather over N "virtual ranks"
 * held as separate buffers in one GPU's memory, plus the LL and LL128 wire
 * formats.  Plain C ABI: device and host pointers, sizes and enums; no C++
 * or PyTorch types.  Library: librra.so (sm_103a).
 *
 * Sources (web pages, cited by title and section):
 *   [ILP] "NCCL collectives, ring all-reduce & launching TP/PP"
 *         (inference-learning-path): "Direct answer", "Deep dive", "Code".
 *   [AIH] "Collective communication: NCCL's algorithms and protocols, and
 *         custom all-reduce in inference frameworks" (ai-infra-handbooks):
 *         "Algorithms: the ways to run one all-reduce", "Protocols: how do
 *         you know the data has arrived", "Reading nccl-tests",
 *         "Common environment variables and debugging", "Exercises" 2 and 3.
 *
 * Conventions shared by every call
 * --------------------------------
 * - A virtual rank r owns one input buffer bufs[r] and one output buffer
 *   outs[r], all device pointers on the current CUDA device.  bufs/outs are
 *   HOST arrays of nranks device pointers; they are read during the call
 *   only (copied into the kernel's parameters), never retained.
 * - Buffers are dense, 1-D, element type `dtype`, little-endian.  Each
 *   pointer must be aligned to the element size; 16-byte aligned buffers
 *   (what cudaMalloc and PyTorch give) take the 128-bit vector path, other
 *   alignments a slower element-wise path with identical results.
 * - The caller owns every buffer.  The library owns only the workspace made
 *   by rra_init() for the device.
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *   default stream), never allocate, never synchronize, and may be captured
 *   into a CUDA graph.  Argument errors are returned synchronously before
 *   any launch.  Errors found on the device (a bounded wait that expired, a
 *   wire flag that never matched) are recorded in the device status word
 *   and read with rra_query_status(), like an asynchronous communicator
 *   error.
 * - Calls that use the workspace (ring, two-shot, LL/LL128 unpack) on one
 *   device must not overlap on the GPU: issue them on one stream or order
 *   them, as with the operations of one communicator.
 * - count == 0 returns RRA_SUCCESS without a launch.
 * - Summation (op RRA_SUM): int32 wraps modulo 2^32; float32 adds in IEEE
 *   round-to-nearest in the order the schedule fixes; bfloat16 is widened
 *   to float32, summed in float32 in that order and rounded to bfloat16
 *   (nearest, ties to even) once, when the final value is stored.
 *
 * Environment (read by the library; none is needed, each overrides a
 * measured default; [AIH] "Common environment variables and debugging"
 * describes NCCL's counterparts)
 * ------------------------------------------------------------------------
 *   RRA_ALGO             schedule for RRA_ALGO_AUTO: ring, one_shot,
 *                        two_shot or tree (instead of the tuning table)
 *   RRA_TUNING_FILE      tuning table read by rra_init (default: tune/
 *                        gb300.txt beside the library)
 *   RRA_TIMEOUT_NS       bound of every device wait (500 ms), unless
 *                        rra_set_timeout_ns() sets one
 *   RRA_MAX_CTAS         CTA budget of every kernel (0: all), unless
 *                        rra_set_max_ctas() sets one
 *   RRA_DEBUG            1: print each call (schedule, grid, status) and
 *                        every CUDA error to stderr
 *   RRA_RING_PROTO       ring links for every buffer: staged, simple or ll
 *                        (per-warp forms); default by size (below)
 *   RRA_RING_LL_STAGED_MAX_BYTES  on 16-byte aligned buffers with 2 ranks
 *                        or more, chunks up to this many bytes take LL
 *                        lines (measured faster there; default 256 KiB from
 *                        3 ranks and 128 KiB at 2, bfloat16 128 KiB),
 *                        larger ones the staged form
 *   RRA_RING_LL_MAX_BYTES  on other buffers, the largest chunk the per-warp
 *                        ring sends as LL lines (64 KiB; larger: Simple)
 *   RRA_RING_CLUSTER     1: the ring on thread-block clusters
 *   RRA_RING_TILE, RRA_RING_G, RRA_RING_K, RRA_RING_STAGES,
 *   RRA_RING_CHANNELS    staged ring: units per message (<= 2368, 1536 for
 *                        bfloat16), messages per step (1-6 by the chunk's
 *                        size per channel), FIFO slots (G+3),
 *                        shared-memory stages, CTAs per rank
 *   RRA_STAGED_SMEM_KB   shared memory for the staged ring's and tree's
 *                        stages (224)
 *   RRA_TREE_TILE, RRA_TREE_G, RRA_TREE_K, RRA_TREE_LAG, RRA_TREE_STAGES,
 *   RRA_TREE_CHANNELS    staged tree: units per message (<= 2048, 1280 for
 *                        bfloat16), tiles per iteration (by size, at most
 *                        24, 12 for bfloat16), FIFO slots (G + 1),
 *                        iterations the broadcast trails the reduction (6),
 *                        stages, CTAs per rank
 *   RRA_TREE_PROTO       ll | staged: the tree's form (default: LL lines
 *                        wherever they fit the workspace's LL region, up to
 *                        RRA_TREE_LL_MAX_BYTES per rank (no limit; bfloat16
 *                        at 2 ranks 1 MiB); the staged tree otherwise)
 *   RRA_TWOSHOT_CLUSTER  1: two-shot on thread-block clusters
 *   RRA_TWOSHOT_CHANNELS CTAs per rank of two-shot
 *   RRA_TWOSHOT_LAG      tiles the two-shot's gather trails its reduce by
 *                        (and between its progress flags): 16 at 8 ranks, 8
 *                        below
 *   RRA_ONESHOT_TMA      1: one-shot with bulk copies through shared memory
 *   RRA_ONESHOT_PER_RANK 1: one-shot reads the n inputs once per rank, as
 *                        n GPUs would (out of place only; in place keeps
 *                        the combined form)
 *   RRA_DIRECT_GRID      grid of one-shot and the direct reduce-scatter and
 *                        all-gather: resident (SMs x occupancy, grid-stride)
 *                        or cover (one trip a thread); default: cover from
 *                        256 MB of floor bytes (one-shot) or 64 MB (the
 *                        others), resident below.  An SM budget keeps the
 *                        resident grid.
 */
#ifndef RRA_H
#define RRA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/** Same object as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st* rra_stream_t;

/** Largest number of virtual ranks (and of LL/LL128 sources) per call. */
#define RRA_MAX_RANKS 8

typedef enum {
  RRA_OK = 0,
  RRA_SUCCESS = RRA_OK,        /* the same value under a second name */
  RRA_ERR_INVALID_ARG = 1,     /* null pointer, bad count, bad enum, misaligned pointer, flag 0 */
  RRA_ERR_UNSUPPORTED = 2,     /* valid but not supported here (e.g. nranks > RRA_MAX_RANKS) */
  RRA_ERR_ALIAS = 3,           /* input and output ranges overlap other than in place */
  RRA_ERR_NOT_INITIALIZED = 4, /* rra_init() was not called for the current device */
  RRA_ERR_CUDA = 5,            /* a CUDA runtime call failed (launch, query) */
  RRA_ERR_TIMEOUT = 6,         /* a bounded device wait expired (see rra_query_status) */
  RRA_ERR_WORKSPACE = 7        /* the workspace of rra_init is too small for the call's FIFO
                                  slots and flags (call rra_init with more workspace_bytes) */
} rra_status_t;

typedef enum { RRA_INT32 = 0, RRA_FLOAT32 = 1, RRA_BFLOAT16 = 2 } rra_dtype_t;

typedef enum { RRA_SUM = 0 } rra_op_t;

/** Schedules ([AIH] "Algorithms").  For reduce-scatter and all-gather,
 *  RRA_ALGO_DIRECT names the direct halves of two-shot (RRA_ALGO_TWO_SHOT
 *  is accepted as a synonym) and RRA_ALGO_RING the ring halves. */
typedef enum {
  RRA_ALGO_AUTO = 0,
  RRA_ALGO_RING = 1,
  RRA_ALGO_ONE_SHOT = 2,
  RRA_ALGO_TWO_SHOT = 3,
  RRA_ALGO_DIRECT = 4,
  /** all-gather only: the GPU's copy engines move the shards
   *  (cudaMemcpyAsync device to device), no SM runs a kernel ([AIH]
   *  "Protocols": transfer methods that use no SMs, like the copy engine). */
  RRA_ALGO_COPY_ENGINE = 5,
  /** all-reduce only: a double binary tree ([AIH] "Algorithms": tree
   *  (double binary tree), reduce up, broadcast down, O(log n) steps,
   *  large messages pipelined in chunks).  Tree 0 is the binary tree in
   *  heap order over the ranks (position p has children 2p+1 and 2p+2,
   *  rank r at position r), tree 1 the same tree over the ranks reversed
   *  (rank r at position n-1-r).  The first part of the message by the
   *  chunk plan for two parts (C = ceil(count/2) rounded up to whole
   *  16-byte vectors) is reduced on tree 0, the rest on tree 1.  A node
   *  sums its own data, then the partial of its child 2p+1, then that of
   *  its child 2p+2; each root's total, rounded once, travels down
   *  unchanged.  Needs 16-byte aligned buffers (else
   *  RRA_ERR_UNSUPPORTED).  Links through the workspace: LL lines for
   *  small messages ("Protocols": LL for small messages), whole-CTA
   *  messages staged by bulk copies for large ones. */
  RRA_ALGO_TREE = 6
} rra_algo_t;

/* ------------------------------------------------------------------------ */
/* set-up                                                                   */
/* ------------------------------------------------------------------------ */

/** Create the per-device state: the workspace (device status word, step
 *  flags, FIFO slots; 64 MiB of them, at most half, hold LL lines only) of
 *  `workspace_bytes` bytes (0 = 256 MiB, at least 1 MiB) on CUDA device
 *  `device`, which becomes current.  Fixed buffers
 *  made once, ahead of the calls, keep every call allocation-free and
 *  graph-capturable, as [AIH] "Exercises" 3 explains for custom
 *  all-reduce.  Calling it again for an initialised device is a no-op that
 *  returns RRA_SUCCESS.  Errors: RRA_ERR_INVALID_ARG (bad device),
 *  RRA_ERR_CUDA (allocation failed). */
rra_status_t rra_init(int device, size_t workspace_bytes);

/** Free the state rra_init made on every device (the pages' communicator
 *  teardown that ends the "init step before calls" of [ILP] "Code").  The
 *  caller must have synchronized every stream that used it; later calls
 *  that need the workspace return RRA_ERR_NOT_INITIALIZED until rra_init
 *  is called again.  Returns RRA_ERR_CUDA if freeing a workspace failed
 *  (the state is dropped all the same). */
rra_status_t rra_finalize(void);

/* ------------------------------------------------------------------------ */
/* collectives                                                              */
/* ------------------------------------------------------------------------ */

/** All-reduce ([ILP] "Direct answer": sum a tensor every rank holds; every
 *  rank ends with the result).  outs[r][i] = SUM_k bufs[k][i] for
 *  i < count, every r.
 *  - bufs[r], outs[r]: count elements each.  In place (outs[r] == bufs[r]
 *    for every r) is allowed; any other overlap is RRA_ERR_ALIAS.
 *  - algo: RING -- n-1 reduce-scatter steps then n-1 all-gather steps over
 *    the N chunks of the chunk plan ([ILP] "Deep dive", [AIH] "Algorithms");
 *    chunk c is summed in the order x_{c+1}, ..., x_{c-1}, x_c.
 *    ONE_SHOT -- every rank's result read directly from all n inputs,
 *    summed in ascending rank order.  TWO_SHOT -- rank r reduces chunk r
 *    (ascending order), then every rank reads the reduced chunks back.
 *    AUTO -- rra_select_algo().
 *  - Chunk plan: chunk length C = ceil(count/n) rounded up to whole
 *    16-byte vectors, chunk c = [min(cC,count), min((c+1)C,count)).
 *  - nranks in [1, RRA_MAX_RANKS]; nranks == 1 copies (or does nothing in
 *    place).
 *  Errors: RRA_ERR_INVALID_ARG, RRA_ERR_UNSUPPORTED, RRA_ERR_ALIAS,
 *  RRA_ERR_NOT_INITIALIZED (RING/TWO_SHOT/AUTO without rra_init),
 *  RRA_ERR_CUDA. */
rra_status_t rra_allreduce(const void* const* bufs, void* const* outs, int nranks, size_t count,
                           rra_dtype_t dtype, rra_op_t op, rra_algo_t algo, rra_stream_t stream);

/** Two-shot all-reduce that allocates nothing.  The pages have no
 *  counterpart: this exists for callers that may not allocate device
 *  memory, and so cannot call rra_init (which calls cudaMalloc for its
 *  workspace).  Examples: a plugin inside a framework whose allocator owns
 *  all device memory, or code under a memory budget that forbids new
 *  allocations after start-up.  It needs no rra_init.
 *  - Same arguments, result and summation order as rra_allreduce with
 *    RRA_ALGO_TWO_SHOT (outs[r][i] = SUM_k bufs[k][i], chunk r reduced in
 *    ascending rank order, then gathered back).  The caller passes the
 *    inputs and outputs; in place is allowed as there.
 *  - Scratch: the kernel's status block, call epoch and step flags live in
 *    a static device array of 16,640 bytes inside librra.so, which every
 *    GPU that loads the library holds until the process exits.  It holds
 *    flags for at most 8 ranks x 16 channels; more than 8 ranks is
 *    RRA_ERR_UNSUPPORTED.  Messages of any size are split over at most 16
 *    channels per rank (fewer under rra_set_max_ctas).
 *  - No cudaMalloc, cudaFree or allocating library routine is called.
 *    The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first
 *    call before any stream capture.
 *  - Every call on a device shares the one array, which keeps the last
 *    call's contents (the flags carry a per-call epoch and need no
 *    clearing; the status block keeps the first device error until
 *    rra_query_status_static reads and clears it).  Calls that overlap on
 *    the GPU -- on two streams without ordering, or together with another
 *    copy of this call -- race on it.
 *  - Device waits are bounded by rra_set_timeout_ns; a wait that expires
 *    ends the kernel early with the outputs partly written, and
 *    rra_query_status_static then returns RRA_ERR_TIMEOUT.  Honours
 *    rra_debug_skip_rank.  Recorded in rra_dump_recent.
 *  Errors: RRA_ERR_INVALID_ARG, RRA_ERR_UNSUPPORTED, RRA_ERR_ALIAS,
 *  RRA_ERR_CUDA.  count == 0 returns RRA_SUCCESS without a launch. */
rra_status_t rra_allreduce_two_shot_static(const void* const* bufs, void* const* outs, int nranks,
                                           size_t count, rra_dtype_t dtype, rra_op_t op,
                                           rra_stream_t stream);

/** Status of rra_allreduce_two_shot_static on the current device, which
 *  allocates nothing either (the pages have no counterpart; it reads the
 *  static scratch array of that entry point, not the workspace of
 *  rra_init).  Synchronizes `stream`, copies the status block to the host
 *  and clears it.  Returns RRA_SUCCESS, the first device error recorded
 *  since the last query (RRA_ERR_TIMEOUT), or RRA_ERR_CUDA.  info (may be
 *  NULL) receives {code, rank, peer, index} as rra_query_status gives it. */
rra_status_t rra_query_status_static(rra_stream_t stream, int32_t info[4]);

/** Reduce-scatter ([ILP] "Direct answer": sum across ranks, each keeps only
 *  its slice).  bufs[r] holds nranks*recvcount elements; outs[r]
 *  (recvcount elements) receives slice r of the sum:
 *  outs[r][i] = SUM_k bufs[k][r*recvcount + i].
 *  - algo RING: chunk c is summed x_{c+1}, ..., x_{c-1}, x_c (the ring's
 *    reduce-scatter half).  DIRECT/TWO_SHOT/AUTO: ascending rank order.
 *  - In place: outs[r] == bufs[r] + r*recvcount elements for every r.
 *  Errors as rra_allreduce; ONE_SHOT is RRA_ERR_INVALID_ARG. */
rra_status_t rra_reduce_scatter(const void* const* bufs, void* const* outs, int nranks,
                                size_t recvcount, rra_dtype_t dtype, rra_op_t op, rra_algo_t algo,
                                rra_stream_t stream);

/** All-gather ([ILP] "Direct answer": each rank holds a shard, every rank
 *  ends with the concatenation).  bufs[r] holds sendcount elements; outs[r]
 *  holds nranks*sendcount: outs[r][q*sendcount + i] = bufs[q][i].
 *  - algo RING: the ring's all-gather half (n-1 forwarding steps).
 *    DIRECT/TWO_SHOT/AUTO: every rank reads every shard directly.
 *    COPY_ENGINE: nranks^2 device-to-device copies on `stream` (no kernel).
 *  - In place: bufs[r] == outs[r] + r*sendcount elements for every r.
 *  The data are copied bit for bit, whatever dtype says.
 *  Errors as rra_allreduce; ONE_SHOT is RRA_ERR_INVALID_ARG. */
rra_status_t rra_all_gather(const void* const* bufs, void* const* outs, int nranks,
                            size_t sendcount, rra_dtype_t dtype, rra_algo_t algo,
                            rra_stream_t stream);

/** All-reduce fused with RMSNorm ([AIH] "Source code": FlashInfer's fused
 *  all-reduce + RMSNorm for tensor-parallel activations).  bufs[r] and
 *  outs[r] hold rows x hidden elements, row-major.  Every rank gets
 *  outs[r][i][j] = s[i][j] * rsqrt(mean_j(s[i][j]^2) + eps) * gamma[j],
 *  where s = SUM_k bufs[k] summed in float32 in ascending rank order (the
 *  one-shot sum).  The normalisation runs in float32; the result is
 *  rounded to dtype once.
 *  - gamma: device pointer, hidden elements of dtype (must not overlap an
 *    output).
 *  - dtype: RRA_FLOAT32 or RRA_BFLOAT16; hidden in [1, 51200]; in place
 *    (outs[r] == bufs[r]) allowed.
 *  Errors: RRA_ERR_INVALID_ARG (int32, null, misaligned, hidden 0),
 *  RRA_ERR_UNSUPPORTED (hidden > 51200, nranks > RRA_MAX_RANKS),
 *  RRA_ERR_ALIAS, RRA_ERR_CUDA.  rows == 0 returns RRA_SUCCESS. */
rra_status_t rra_allreduce_rmsnorm(const void* const* bufs, void* const* outs, int nranks,
                                   size_t rows, size_t hidden, const void* gamma, float eps,
                                   rra_dtype_t dtype, rra_stream_t stream);

/* ------------------------------------------------------------------------ */
/* LL and LL128 wire formats ([AIH] "Protocols")                            */
/* ------------------------------------------------------------------------ */

/** Bytes of LL wire for a payload: 8 * ceil(payload_bytes / 4).  LL: every
 *  8-byte line holds 4 bytes of data and a 4-byte flag (50% efficiency). */
size_t rra_ll_wire_bytes(size_t payload_bytes);

/** Bytes of LL128 wire: 128 * ceil(payload_bytes / 120).  LL128: every
 *  128-byte line holds 120 bytes of data and an 8-byte flag (93.75%). */
size_t rra_ll128_wire_bytes(size_t payload_bytes);

/** LL pack: line i of `wire` (device, 16-byte aligned,
 *  rra_ll_wire_bytes(payload_bytes) bytes) gets payload bytes [4i, 4i+4) in
 *  its bytes 0..3 (zero past the payload's end) and `flag` (little-endian)
 *  in bytes 4..7.  Lines are written with single 16-byte stores, so a
 *  line's data and flag become visible together.  flag must be nonzero (0
 *  marks an empty line); callers use a step counter 1, 2, ...  `payload`
 *  is a device pointer (any alignment).  Errors: RRA_ERR_INVALID_ARG. */
rra_status_t rra_ll_pack(const void* payload, size_t payload_bytes, void* wire, uint32_t flag,
                         rra_stream_t stream);

/** LL unpack-and-reduce: for every line, poll each of the nsrc wires until
 *  its flag equals expected_flag (a bounded wait, rra_set_timeout_ns), then
 *  write the element-wise SUM of the nsrc data words, sources in ascending
 *  order, to out (payload_bytes bytes, a whole number of dtype elements).
 *  nsrc == 1 is a plain unpack.  wires: host array of nsrc device pointers
 *  (16-byte aligned).  A line whose flag never matches ends the wait with
 *  RRA_ERR_TIMEOUT in the status word: info = {code, source, -1, line}.
 *  Needs rra_init().  Errors: RRA_ERR_INVALID_ARG, RRA_ERR_UNSUPPORTED,
 *  RRA_ERR_NOT_INITIALIZED. */
rra_status_t rra_ll_unpack(const void* const* wires, int nsrc, void* out, size_t payload_bytes,
                           rra_dtype_t dtype, rra_op_t op, uint32_t expected_flag,
                           rra_stream_t stream);

/** LL128 pack: line j (128 bytes) of `wire` gets payload bytes
 *  [120j, 120j+120) in bytes 0..119 (zero past the end) and `flag` as a
 *  little-endian uint64 in bytes 120..127.  A warp writes four lines with
 *  32 16-byte stores.  Other rules as rra_ll_pack. */
rra_status_t rra_ll128_pack(const void* payload, size_t payload_bytes, void* wire, uint64_t flag,
                            rra_stream_t stream);

/** LL128 unpack-and-reduce: a warp reads four lines of each source (one
 *  16-byte load per lane), checks the four flags across the warp, and on a
 *  match sums the 120 data bytes of every line over the sources (ascending
 *  order).  Other rules as rra_ll_unpack. */
rra_status_t rra_ll128_unpack(const void* const* wires, int nsrc, void* out, size_t payload_bytes,
                              rra_dtype_t dtype, rra_op_t op, uint64_t expected_flag,
                              rra_stream_t stream);

/* ------------------------------------------------------------------------ */
/* status, selection, configuration                                         */
/* ------------------------------------------------------------------------ */

/** The asynchronous error of the calls issued so far, as NCCL reports an
 *  asynchronous communicator error ([AIH] "Common environment variables
 *  and debugging": a collective that hangs or fails is found from the
 *  device side, not from the launch).  Synchronize `stream`, then read and
 *  clear the current device's status word.  Returns RRA_SUCCESS, the
 *  recorded device error (RRA_ERR_TIMEOUT) or RRA_ERR_CUDA if the stream
 *  itself failed.  info (may be NULL) receives {code, rank, peer, index}:
 *  the rank (or LL source) whose wait expired, the rank it waited for (-1
 *  if none) and the step (ring, two-shot) or line (LL, LL128) index. */
rra_status_t rra_query_status(rra_stream_t stream, int32_t info[4]);

/** The schedule AUTO uses for an all-reduce of bytes_per_rank bytes per
 *  rank: from the measured table (rra_load_tuning; the table shipped
 *  beside the library is loaded by rra_init) when it has an entry for
 *  nranks and dtype; else from the alpha-beta cost model of [AIH]
 *  "Algorithms" with alpha and beta fitted on this GPU (the table's "ab"
 *  lines): the schedule with the least alpha * syncs(n) + beta * n * S,
 *  syncs being 2(n-1) for the ring, 1 for one-shot, 2 for two-shot and
 *  2 ceil(log2 n) for the tree; with no table loaded, one-shot (on one GPU
 *  every schedule moves the same 2nS bytes and one-shot has the fewest
 *  syncs).  AUTO never runs the tree on buffers that are not 16-byte
 *  aligned.  Never returns RRA_ALGO_AUTO. */
rra_algo_t rra_select_algo(int nranks, size_t bytes_per_rank, rra_dtype_t dtype);

/** Load a tuning table ([AIH] "Algorithms": the alpha-beta crossovers are
 *  only illustrative and must be measured on one's own machine; this is
 *  where the measured ones go): text lines "nranks dtype log2_bytes algo"
 *  (dtype int32|float32|bfloat16, algo ring|one_shot|two_shot|tree), and
 *  prior lines "ab dtype algo alpha_us beta_us_per_MiB" (alpha per
 *  synchronization, beta per MiB of nranks x bytes_per_rank); '#' starts a
 *  comment.  The entry with the largest log2_bytes <= ceil(log2(bytes))
 *  for (nranks, dtype) wins.  NULL clears the table.  Errors:
 *  RRA_ERR_INVALID_ARG (unreadable or malformed file; the old table stays). */
rra_status_t rra_load_tuning(const char* path);

/** Upper bound, in nanoseconds of %globaltimer, on every device-side wait
 *  (ring, tree and two-shot step flags, LL/LL128 line flags).  [AIH]
 *  "Common environment variables and debugging" describes collectives that
 *  wait forever for a rank that never arrives; here every such wait ends
 *  after this bound with RRA_ERR_TIMEOUT in the status word.  Default 500
 *  ms or RRA_TIMEOUT_NS from the environment; 0 restores the default.
 *  Also bounds the waits of rra_allreduce_two_shot_static. */
void rra_set_timeout_ns(uint64_t ns);

/** SM budget ([AIH] "Protocols": each channel is a CUDA block, and
 *  communication kernels compete with compute for SMs): at most
 *  `max_ctas` CTAs per launch (0 = no limit, the default, or RRA_MAX_CTAS
 *  from the environment).  Streaming kernels shrink their grid and loop
 *  longer; ring and two-shot use at most max_ctas / nranks channels (at
 *  least one). */
void rra_set_max_ctas(int max_ctas);

/** Fault injection for tests: virtual rank `rank` posts no step flag in the
 *  following ring, two-shot (also rra_allreduce_two_shot_static) and tree
 *  calls (-1 turns it off), so its peers' waits expire with RRA_ERR_TIMEOUT
 *  naming it as `peer`.  The GPU stays usable. */
void rra_debug_skip_rank(int rank);

/** Static text for a status code, for the error reports [AIH] "Common
 *  environment variables and debugging" asks to read first when a
 *  collective fails. */
const char* rra_status_string(rra_status_t status);

/** Flight recorder ([AIH] "Common environment variables and debugging":
 *  a record of each rank's recent collectives): writes the last calls
 *  (sequence number, call, algo, nranks, count, dtype, grid, result), one
 *  per line, oldest first, into buf (NUL-terminated, truncated to len).
 *  Returns the number of calls written. */
int rra_dump_recent(char* buf, size_t len);

#ifdef __cplusplus
}
#endif

#endif /* RRA_H */
