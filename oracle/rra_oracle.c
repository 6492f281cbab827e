/*
 * rra_oracle.c -- plain, slow CPU oracle for the virtual-rank collectives.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load it (through oracle/__init__.py).  It shares no code,
 * header, table or helper with the CUDA path.
 *
 * Every schedule is simulated literally, rank by rank and step by step, over
 * host arrays, with per-rank staging buffers and byte counters.  Nothing is
 * blocked, fused or reordered beyond what the schedule itself states.
 *
 * Sources (web pages; cited by title and section):
 *   [ILP]  "NCCL collectives, ring all-reduce & launching TP/PP"
 *          (inference-learning-path), sections "Direct answer", "Deep dive".
 *   [AIH]  "Collective communication: NCCL's algorithms and protocols, and
 *          custom all-reduce in inference frameworks" (ai-infra-handbooks),
 *          sections "Algorithms: the ways to run one all-reduce",
 *          "Protocols: how do you know the data has arrived",
 *          "Reading nccl-tests", "Exercises".
 *
 * Arithmetic (the pages leave it open; the readings taken):
 *   int32    : added as uint32, so overflow wraps modulo 2^32.
 *   float32  : IEEE single, round-to-nearest, in the order each schedule
 *              fixes.  Build without -ffast-math and with -ffp-contract=off.
 *   bfloat16 : decoded exactly to float32, accumulated in float32 in the
 *              schedule's order, rounded once to bfloat16 (round to nearest,
 *              ties to even) when the final value is stored.  Ring partial
 *              sums travel as float32 and are never re-rounded per step.
 *
 * Byte counters: recv[r] counts the payload bytes rank r obtains from other
 * ranks (received or read); sent[r] counts the bytes other ranks obtain from
 * rank r.  Payload bytes are element count x element size of the data type,
 * also for the float32 partials that carry bfloat16 data.
 */
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#define ORC_INT32 0
#define ORC_FLOAT32 1
#define ORC_BFLOAT16 2

#define ORC_OK 0
#define ORC_EINVAL -1
#define ORC_ENOMEM -2

/* ------------------------------------------------------------------------ */
/* element types                                                            */
/* ------------------------------------------------------------------------ */

static size_t elem_size(int dt) {
  return dt == ORC_BFLOAT16 ? 2u : 4u;
}

/* bfloat16 -> float32 is exact: the 16 bits are the high half of the float. */
float orc_bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* float32 -> bfloat16, round to nearest, ties to even, written from the
 * IEEE-754 definition on the float's bit pattern: keep the high 16 bits,
 * look at the 16 discarded bits, round up when they exceed half an ulp or
 * equal half an ulp with an odd kept part.  A carry out of the mantissa
 * moves into the exponent, which is what IEEE rounding asks (the largest
 * finite values round up to infinity).  NaN maps to the quiet NaN 0x7FC0. */
uint16_t orc_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
    return (uint16_t)0x7FC0u;
  uint32_t kept = u >> 16;
  uint32_t dropped = u & 0xFFFFu;
  if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
    kept += 1u;
  return (uint16_t)kept;
}

/* Accumulators are 4 bytes wide: uint32 for int32, float for the others. */
static void acc_load(int dt, const void* x, size_t off, size_t len, void* acc) {
  for (size_t i = 0; i < len; ++i) {
    if (dt == ORC_INT32) {
      uint32_t v;
      memcpy(&v, (const char*)x + 4 * (off + i), 4);
      ((uint32_t*)acc)[i] = v;
    } else if (dt == ORC_FLOAT32) {
      float v;
      memcpy(&v, (const char*)x + 4 * (off + i), 4);
      ((float*)acc)[i] = v;
    } else {
      uint16_t h;
      memcpy(&h, (const char*)x + 2 * (off + i), 2);
      ((float*)acc)[i] = orc_bf16_to_f32(h);
    }
  }
}

/* acc[i] = acc[i] (+) x[off+i]: the running sum comes first, the newly read
 * value second, so a left fold over ranks is exactly the loop order. */
static void acc_add(int dt, void* acc, const void* x, size_t off, size_t len) {
  for (size_t i = 0; i < len; ++i) {
    if (dt == ORC_INT32) {
      uint32_t v;
      memcpy(&v, (const char*)x + 4 * (off + i), 4);
      ((uint32_t*)acc)[i] = ((uint32_t*)acc)[i] + v;
    } else if (dt == ORC_FLOAT32) {
      float v;
      memcpy(&v, (const char*)x + 4 * (off + i), 4);
      ((float*)acc)[i] = ((float*)acc)[i] + v;
    } else {
      uint16_t h;
      memcpy(&h, (const char*)x + 2 * (off + i), 2);
      ((float*)acc)[i] = ((float*)acc)[i] + orc_bf16_to_f32(h);
    }
  }
}

/* y[off+i] = narrow(acc[i]); bfloat16 is rounded here, once. */
static void acc_store(int dt, const void* acc, void* y, size_t off, size_t len) {
  for (size_t i = 0; i < len; ++i) {
    if (dt == ORC_INT32) {
      memcpy((char*)y + 4 * (off + i), (const uint32_t*)acc + i, 4);
    } else if (dt == ORC_FLOAT32) {
      memcpy((char*)y + 4 * (off + i), (const float*)acc + i, 4);
    } else {
      uint16_t h = orc_f32_to_bf16(((const float*)acc)[i]);
      memcpy((char*)y + 2 * (off + i), &h, 2);
    }
  }
}

static void tally(uint64_t* ctr, int r, uint64_t bytes) {
  if (ctr) ctr[r] += bytes;
}

static int mod(int a, int n) {
  int m = a % n;
  return m < 0 ? m + n : m;
}

/* ------------------------------------------------------------------------ */
/* chunk plan                                                               */
/* ------------------------------------------------------------------------ */

/* [ILP] "Deep dive": the ring "pipelines the data in N chunks".  The pages do
 * not say where the chunk edges fall when n does not divide count; the
 * reading taken: chunk length C = ceil(count/n) rounded up to a whole number
 * of 16-byte vectors (V = 16/elem elements), chunk c = [min(cC, count),
 * min((c+1)C, count)).  Trailing chunks may be short or empty.
 * bounds[] receives n+1 entries. */
int orc_chunk_plan(int n, size_t count, int dt, size_t* bounds) {
  if (n < 1 || !bounds) return ORC_EINVAL;
  size_t v = 16u / elem_size(dt);
  size_t per = (count + (size_t)n - 1u) / (size_t)n;
  size_t c_len = ((per + v - 1u) / v) * v;
  for (int c = 0; c <= n; ++c) {
    size_t b = (size_t)c * c_len;
    bounds[c] = b < count ? b : count;
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* ring: reduce-scatter half and all-gather half                            */
/* ------------------------------------------------------------------------ */

/* The ring reduce-scatter of [AIH] "Algorithms" (ring: n-1 reduce-scatter
 * steps, each GPU sending and receiving (n-1)/n of the data per phase) and
 * [ILP] "Direct answer" (ring all-reduce = reduce-scatter + all-gather).
 *
 * Chunk c of rank r's input is in[r][ibase[c] .. ibase[c] + len[c]).
 * Step s = 0..n-2: every rank r sends the partial it holds, which belongs to
 * chunk (r-s-1) mod n, to rank r+1; the receiver adds its own slice of that
 * chunk to what arrived.  Before step 0 rank r holds its own slice of chunk
 * (r-1) mod n.  After the last step rank r holds chunk r, summed in the
 * order x_{r+1}, x_{r+2}, ..., x_{r-1}, x_r (indices mod n).  The reduced
 * chunk r is written to out[r][obase[r] ..]. */
static int ring_reduce_scatter(int n, int dt, const size_t* ibase, const size_t* len,
                               const void* const* in, void* const* out, const size_t* obase,
                               uint64_t* sent, uint64_t* recv) {
  if (n < 1) return ORC_EINVAL;
  size_t e = elem_size(dt);
  size_t cmax = 0;
  for (int c = 0; c < n; ++c)
    if (len[c] > cmax) cmax = len[c];
  /* hold[r]: the partial rank r is about to send; inbox[r]: what it received */
  void** hold = (void**)calloc((size_t)n, sizeof(void*));
  void** inbox = (void**)calloc((size_t)n, sizeof(void*));
  int rc = ORC_OK;
  if (!hold || !inbox) { rc = ORC_ENOMEM; goto done; }
  for (int r = 0; r < n; ++r) {
    hold[r] = malloc(cmax * 4 + 4);
    inbox[r] = malloc(cmax * 4 + 4);
    if (!hold[r] || !inbox[r]) { rc = ORC_ENOMEM; goto done; }
  }
  for (int r = 0; r < n; ++r) {
    int c = mod(r - 1, n);
    acc_load(dt, in[r], ibase[c], len[c], hold[r]);
  }
  for (int s = 0; s <= n - 2; ++s) {
    /* deliver: rank r -> rank r+1, chunk (r-s-1) mod n */
    for (int r = 0; r < n; ++r) {
      int dst = mod(r + 1, n);
      int c = mod(r - s - 1, n);
      memcpy(inbox[dst], hold[r], len[c] * 4);
      tally(sent, r, len[c] * e);
      tally(recv, dst, len[c] * e);
    }
    /* reduce at the receiver: received partial first, own slice second */
    for (int r = 0; r < n; ++r) {
      int c = mod(r - 1 - s - 1, n); /* the chunk rank r-1 sent in step s */
      memcpy(hold[r], inbox[r], len[c] * 4);
      acc_add(dt, hold[r], in[r], ibase[c], len[c]);
    }
  }
  for (int r = 0; r < n; ++r) {
    /* n == 1: no step ran and hold[0] is rank 0's own chunk 0 */
    acc_store(dt, hold[r], out[r], obase[r], len[r]);
  }
done:
  if (hold)
    for (int r = 0; r < n; ++r) free(hold[r]);
  if (inbox)
    for (int r = 0; r < n; ++r) free(inbox[r]);
  free(hold);
  free(inbox);
  return rc;
}

/* The ring all-gather of [AIH] "Algorithms" (n-1 all-gather steps) and [ILP]
 * "Direct answer".  Rank r starts holding chunk r, already stored at
 * out[r][obase[r] ..].  Step s = 0..n-2: rank r forwards chunk (r-s) mod n to
 * rank r+1, which stores it into its own output at obase of that chunk and
 * forwards it in the next step.  Chunk c has len[c] elements. */
static int ring_all_gather(int n, int dt, const size_t* obase, const size_t* len,
                           void* const* out, uint64_t* sent, uint64_t* recv) {
  if (n < 1) return ORC_EINVAL;
  size_t e = elem_size(dt);
  size_t cmax = 0;
  for (int c = 0; c < n; ++c)
    if (len[c] > cmax) cmax = len[c];
  char** hold = (char**)calloc((size_t)n, sizeof(char*));
  char** inbox = (char**)calloc((size_t)n, sizeof(char*));
  int rc = ORC_OK;
  if (!hold || !inbox) { rc = ORC_ENOMEM; goto done; }
  for (int r = 0; r < n; ++r) {
    hold[r] = (char*)malloc(cmax * e + 4);
    inbox[r] = (char*)malloc(cmax * e + 4);
    if (!hold[r] || !inbox[r]) { rc = ORC_ENOMEM; goto done; }
  }
  for (int r = 0; r < n; ++r)
    memcpy(hold[r], (char*)out[r] + obase[r] * e, len[r] * e);
  for (int s = 0; s <= n - 2; ++s) {
    for (int r = 0; r < n; ++r) {
      int dst = mod(r + 1, n);
      int c = mod(r - s, n);
      memcpy(inbox[dst], hold[r], len[c] * e);
      tally(sent, r, len[c] * e);
      tally(recv, dst, len[c] * e);
    }
    for (int r = 0; r < n; ++r) {
      int c = mod(r - 1 - s, n); /* the chunk rank r-1 forwarded in step s */
      memcpy((char*)out[r] + obase[c] * e, inbox[r], len[c] * e);
      memcpy(hold[r], inbox[r], len[c] * e);
    }
  }
done:
  if (hold)
    for (int r = 0; r < n; ++r) free(hold[r]);
  if (inbox)
    for (int r = 0; r < n; ++r) free(inbox[r]);
  free(hold);
  free(inbox);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* all-reduce schedules                                                     */
/* ------------------------------------------------------------------------ */

/* Ring all-reduce: [ILP] "Direct answer" (reduce-scatter then all-gather)
 * and [AIH] "Algorithms" (n-1 steps of each, 2(n-1)/n S sent and received
 * per GPU), over the N chunks of orc_chunk_plan.  Rank c ends the
 * reduce-scatter with chunk c; the all-gather then spreads it. */
int orc_allreduce_ring(int n, size_t count, int dt, const void* const* in, void* const* out,
                       uint64_t* sent, uint64_t* recv) {
  if (n < 1 || n > 64) return ORC_EINVAL;
  size_t b[65], len[64];
  orc_chunk_plan(n, count, dt, b);
  for (int c = 0; c < n; ++c) len[c] = b[c + 1] - b[c];
  int rc = ring_reduce_scatter(n, dt, b, len, in, out, b, sent, recv);
  if (rc) return rc;
  return ring_all_gather(n, dt, b, len, out, sent, recv);
}

/* One-shot: [AIH] "Algorithms" -- each GPU reads the full data of the other
 * n-1 GPUs directly and sums locally; one synchronization; (n-1) S read per
 * GPU.  Every rank sums in ascending rank order 0..n-1, so all ranks hold
 * the same bits (all-reduce leaves every GPU with the result, [ILP]). */
int orc_allreduce_oneshot(int n, size_t count, int dt, const void* const* in, void* const* out,
                          uint64_t* sent, uint64_t* recv) {
  if (n < 1) return ORC_EINVAL;
  size_t e = elem_size(dt);
  void* acc = malloc(count * 4 + 4);
  if (!acc) return ORC_ENOMEM;
  for (int r = 0; r < n; ++r) {
    acc_load(dt, in[0], 0, count, acc);
    for (int k = 1; k < n; ++k) acc_add(dt, acc, in[k], 0, count);
    for (int k = 0; k < n; ++k)
      if (k != r) {
        tally(recv, r, count * e);
        tally(sent, k, count * e);
      }
    acc_store(dt, acc, out[r], 0, count);
  }
  free(acc);
  return ORC_OK;
}

/* Direct reduce-scatter step shared by two-shot and the direct RS: rank r
 * reads its 1/n slice (chunk r) from every rank and sums it in ascending
 * rank order.  Chunk c of a rank's input sits at ibase[c]; the result goes to
 * out[r][obase[r] ..]. */
static int direct_reduce(int n, int dt, const size_t* ibase, const size_t* len,
                         const void* const* in, void* const* out, const size_t* obase,
                         uint64_t* sent, uint64_t* recv) {
  size_t e = elem_size(dt);
  size_t cmax = 0;
  for (int c = 0; c < n; ++c)
    if (len[c] > cmax) cmax = len[c];
  void* acc = malloc(cmax * 4 + 4);
  if (!acc) return ORC_ENOMEM;
  for (int r = 0; r < n; ++r) {
    acc_load(dt, in[0], ibase[r], len[r], acc);
    for (int k = 1; k < n; ++k) acc_add(dt, acc, in[k], ibase[r], len[r]);
    for (int k = 0; k < n; ++k)
      if (k != r) {
        tally(recv, r, len[r] * e);
        tally(sent, k, len[r] * e);
      }
    acc_store(dt, acc, out[r], obase[r], len[r]);
  }
  free(acc);
  return ORC_OK;
}

/* Direct all-gather step: rank r reads every peer's chunk q from where that
 * peer holds it (src[q] + sbase[q]) into out[r][obase[q] ..]. */
static void direct_gather(int n, int dt, const size_t* len, const void* const* src,
                          const size_t* sbase, void* const* out, const size_t* obase,
                          uint64_t* sent, uint64_t* recv) {
  size_t e = elem_size(dt);
  for (int r = 0; r < n; ++r)
    for (int q = 0; q < n; ++q) {
      if (q == r) continue;
      memcpy((char*)out[r] + obase[q] * e, (const char*)src[q] + sbase[q] * e, len[q] * e);
      tally(recv, r, len[q] * e);
      tally(sent, q, len[q] * e);
    }
}

/* Two-shot: [AIH] "Algorithms" -- first each GPU reads only its 1/n of the
 * other GPUs' data and sums it (a reduce-scatter), then reads the sums back
 * (an all-gather); two synchronizations; 2(n-1)/n S read per GPU.  Slices
 * are the chunks of orc_chunk_plan, summed in ascending rank order. */
int orc_allreduce_twoshot(int n, size_t count, int dt, const void* const* in, void* const* out,
                          uint64_t* sent, uint64_t* recv) {
  if (n < 1 || n > 64) return ORC_EINVAL;
  size_t b[65], len[64];
  orc_chunk_plan(n, count, dt, b);
  for (int c = 0; c < n; ++c) len[c] = b[c + 1] - b[c];
  int rc = direct_reduce(n, dt, b, len, in, out, b, sent, recv);
  if (rc) return rc;
  /* phase 2 reads the reduced slices where phase 1 left them */
  direct_gather(n, dt, len, (const void* const*)out, b, out, b, sent, recv);
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* standalone reduce-scatter and all-gather                                 */
/* ------------------------------------------------------------------------ */

/* Reduce-scatter ([ILP] "Direct answer": sum across GPUs, each keeps only its
 * slice of the sum).  in[r] holds n*recvcount elements; slice c is
 * [c*recvcount, (c+1)*recvcount); out[r] (recvcount elements) receives the
 * reduced slice r.  Ring order as in ring_reduce_scatter. */
int orc_reduce_scatter_ring(int n, size_t recvcount, int dt, const void* const* in,
                            void* const* out, uint64_t* sent, uint64_t* recv) {
  if (n < 1 || n > 64) return ORC_EINVAL;
  size_t ib[64], len[64], ob[64];
  for (int c = 0; c < n; ++c) {
    ib[c] = (size_t)c * recvcount;
    len[c] = recvcount;
    ob[c] = 0;
  }
  return ring_reduce_scatter(n, dt, ib, len, in, out, ob, sent, recv);
}

/* Direct reduce-scatter (the first half of two-shot): ascending rank order. */
int orc_reduce_scatter_direct(int n, size_t recvcount, int dt, const void* const* in,
                              void* const* out, uint64_t* sent, uint64_t* recv) {
  if (n < 1 || n > 64) return ORC_EINVAL;
  size_t ib[64], len[64], ob[64];
  for (int c = 0; c < n; ++c) {
    ib[c] = (size_t)c * recvcount;
    len[c] = recvcount;
    ob[c] = 0;
  }
  return direct_reduce(n, dt, ib, len, in, out, ob, sent, recv);
}

/* All-gather ([ILP] "Direct answer": each GPU holds a shard, every GPU ends
 * with the full concatenation).  in[r] holds sendcount elements; out[r]
 * (n*sendcount) receives shard q at [q*sendcount, (q+1)*sendcount).  The own
 * shard is a local copy and not counted as traffic. */
int orc_all_gather_ring(int n, size_t sendcount, int dt, const void* const* in,
                        void* const* out, uint64_t* sent, uint64_t* recv) {
  if (n < 1 || n > 64) return ORC_EINVAL;
  size_t e = elem_size(dt);
  size_t ob[64], len[64];
  for (int c = 0; c < n; ++c) {
    ob[c] = (size_t)c * sendcount;
    len[c] = sendcount;
  }
  for (int r = 0; r < n; ++r) memcpy((char*)out[r] + ob[r] * e, in[r], sendcount * e);
  return ring_all_gather(n, dt, ob, len, out, sent, recv);
}

/* Direct all-gather (the second half of two-shot): every rank reads each
 * peer's shard from the peer's input. */
int orc_all_gather_direct(int n, size_t sendcount, int dt, const void* const* in,
                          void* const* out, uint64_t* sent, uint64_t* recv) {
  if (n < 1 || n > 64) return ORC_EINVAL;
  size_t e = elem_size(dt);
  size_t ob[64], len[64], sb[64];
  for (int c = 0; c < n; ++c) {
    ob[c] = (size_t)c * sendcount;
    len[c] = sendcount;
    sb[c] = 0;
  }
  for (int r = 0; r < n; ++r) memcpy((char*)out[r] + ob[r] * e, in[r], sendcount * e);
  direct_gather(n, dt, len, in, sb, out, ob, sent, recv);
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* LL and LL128 wire formats                                                */
/* ------------------------------------------------------------------------ */

/* [AIH] "Protocols": LL -- every 8 bytes hold 4 bytes of data and 4 bytes of
 * flag, and the receiver polls the flag.  Layout read here: line i carries
 * payload bytes [4i, 4i+4) in its bytes 0..3 (zero past the payload's end)
 * and the flag as a little-endian uint32 in bytes 4..7. */
size_t orc_ll_wire_bytes(size_t payload_bytes) {
  return 8u * ((payload_bytes + 3u) / 4u);
}

void orc_ll_pack(const void* payload, size_t payload_bytes, void* wire, uint32_t flag) {
  const unsigned char* p = (const unsigned char*)payload;
  unsigned char* w = (unsigned char*)wire;
  size_t lines = (payload_bytes + 3u) / 4u;
  for (size_t i = 0; i < lines; ++i) {
    for (int b = 0; b < 4; ++b) {
      size_t src = 4u * i + (size_t)b;
      w[8u * i + (size_t)b] = src < payload_bytes ? p[src] : 0u;
    }
    for (int b = 0; b < 4; ++b) w[8u * i + 4u + (size_t)b] = (unsigned char)(flag >> (8 * b));
  }
}

/* [AIH] "Protocols": LL128 -- every 128 bytes hold 120 bytes of data and 8
 * bytes of flag.  Layout read here: line j carries payload bytes
 * [120j, 120j+120) in its bytes 0..119 (zero past the end) and the flag as a
 * little-endian uint64 in bytes 120..127. */
size_t orc_ll128_wire_bytes(size_t payload_bytes) {
  return 128u * ((payload_bytes + 119u) / 120u);
}

void orc_ll128_pack(const void* payload, size_t payload_bytes, void* wire, uint64_t flag) {
  const unsigned char* p = (const unsigned char*)payload;
  unsigned char* w = (unsigned char*)wire;
  size_t lines = (payload_bytes + 119u) / 120u;
  for (size_t j = 0; j < lines; ++j) {
    for (int b = 0; b < 120; ++b) {
      size_t src = 120u * j + (size_t)b;
      w[128u * j + (size_t)b] = src < payload_bytes ? p[src] : 0u;
    }
    for (int b = 0; b < 8; ++b) w[128u * j + 120u + (size_t)b] = (unsigned char)(flag >> (8 * b));
  }
}

/* Unpack-and-reduce shared by both formats: for each line, every source's
 * flag must equal the expected one (the receiver learns from the flag that
 * the line has arrived; the oracle reports the first line whose flag is
 * wrong instead of waiting).  The data bytes of all sources are then summed
 * element by element in ascending source order and the first payload_bytes
 * bytes are written out.  Returns -1 when every flag matched, else the index
 * of the first line (in line order, sources checked 0..nsrc-1) whose flag
 * differs; out is then left partly written. */
static long long unpack_reduce(const void* const* wires, int nsrc, void* out, size_t payload_bytes,
                               int dt, size_t line_bytes, size_t data_bytes, int flag_bytes,
                               uint64_t expected) {
  size_t e = elem_size(dt);
  size_t lines = (payload_bytes + data_bytes - 1u) / data_bytes;
  size_t per_line = data_bytes / e;
  unsigned char* o = (unsigned char*)out;
  unsigned char line_out[128];
  uint32_t acc[64];
  for (size_t j = 0; j < lines; ++j) {
    for (int k = 0; k < nsrc; ++k) {
      const unsigned char* w = (const unsigned char*)wires[k] + j * line_bytes;
      uint64_t f = 0;
      for (int b = 0; b < flag_bytes; ++b) f |= (uint64_t)w[data_bytes + (size_t)b] << (8 * b);
      if (f != expected) return (long long)j;
    }
    acc_load(dt, (const unsigned char*)wires[0] + j * line_bytes, 0, per_line, acc);
    for (int k = 1; k < nsrc; ++k)
      acc_add(dt, acc, (const unsigned char*)wires[k] + j * line_bytes, 0, per_line);
    acc_store(dt, acc, line_out, 0, per_line);
    size_t lo = j * data_bytes;
    size_t take = payload_bytes - lo < data_bytes ? payload_bytes - lo : data_bytes;
    memcpy(o + lo, line_out, take);
  }
  return -1;
}

long long orc_ll_unpack(const void* const* wires, int nsrc, void* out, size_t payload_bytes, int dt,
                        uint32_t expected_flag) {
  if (nsrc < 1 || payload_bytes % elem_size(dt)) return -2;
  return unpack_reduce(wires, nsrc, out, payload_bytes, dt, 8u, 4u, 4, expected_flag);
}

long long orc_ll128_unpack(const void* const* wires, int nsrc, void* out, size_t payload_bytes,
                           int dt, uint64_t expected_flag) {
  if (nsrc < 1 || payload_bytes % elem_size(dt)) return -2;
  return unpack_reduce(wires, nsrc, out, payload_bytes, dt, 128u, 120u, 8, expected_flag);
}

/* ------------------------------------------------------------------------ */
/* fused all-reduce + RMSNorm                                               */
/* ------------------------------------------------------------------------ */

/* "Collective communication: NCCL's algorithms and protocols, ...",
 * section "Source code", names FlashInfer's fused all-reduce + RMSNorm for
 * the tensor-parallel activations [tokens, hidden]; the page gives no
 * formula.  Reading taken: the all-reduce is the one-shot sum (float32,
 * ascending rank order), then each row is normalised by its root mean
 * square: y[i][j] = s[i][j] / sqrt(mean_j(s[i][j]^2) + eps) * gamma[j].
 * The normalisation runs in double here (no precision is fixed for it) and
 * the result is rounded to the element type once (float32 first, then
 * bfloat16 for bfloat16 output).  Every rank receives the same rows.
 * gamma has the element type; int32 is not accepted. */
int orc_allreduce_rmsnorm(int n, size_t rows, size_t hidden, int dt, const void* const* in,
                          const void* gamma, double eps, void* const* out) {
  if (n < 1 || dt == ORC_INT32) return ORC_EINVAL;
  float* s = (float*)malloc(hidden * 4 + 4);
  float* g = (float*)malloc(hidden * 4 + 4);
  float* y = (float*)malloc(hidden * 4 + 4);
  if (!s || !g || !y) {
    free(s);
    free(g);
    free(y);
    return ORC_ENOMEM;
  }
  acc_load(dt, gamma, 0, hidden, g);
  for (size_t i = 0; i < rows; ++i) {
    acc_load(dt, in[0], i * hidden, hidden, s);
    for (int k = 1; k < n; ++k) acc_add(dt, s, in[k], i * hidden, hidden);
    double ss = 0.0;
    for (size_t j = 0; j < hidden; ++j) ss += (double)s[j] * (double)s[j];
    const double inv = 1.0 / sqrt(ss / (double)hidden + eps);
    for (size_t j = 0; j < hidden; ++j) y[j] = (float)((double)s[j] * inv * (double)g[j]);
    for (int r = 0; r < n; ++r) acc_store(dt, y, out[r], i * hidden, hidden);
  }
  free(s);
  free(g);
  free(y);
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* tree all-reduce                                                          */
/* ------------------------------------------------------------------------ */

/* "Collective communication: NCCL's algorithms and protocols, ...",
 * section "Algorithms": the tree is a double binary tree -- reduce up the
 * tree, then broadcast down it, in O(log n) steps, with large messages
 * pipelined in chunks.  The page fixes neither the two trees' shapes, nor
 * how the data is shared between them, nor the order a node adds its
 * inputs.  The reading taken:
 *   - tree 0 is the binary tree in heap order over the ranks (position p
 *     has children 2p+1 and 2p+2 and parent (p-1)/2), rank r at position
 *     r; tree 1 is the same tree over the ranks in reverse order, rank r at
 *     position n-1-r.  With n even, the ranks that are inner nodes of one
 *     tree (positions below n/2) are the leaves of the other, so no rank is
 *     an inner node of both; with n odd, rank (n-1)/2 is a leaf of both.
 *   - the message is split in two by the chunk plan for two parts: the
 *     first part (elements [0, H)) is reduced and broadcast on tree 0, the
 *     second ([H, count)) on tree 1.
 *   - a node's partial is its own data, then the partial of its child at
 *     position 2p+1, then that of its child at 2p+2:
 *     p = (x (+) p_{2p+1}) (+) p_{2p+2}, missing children skipped.  The
 *     root's total is rounded once and handed down unchanged, so every rank
 *     gets the same bits.
 * Byte counters: in each tree every non-root node sends its partial up once
 * and receives the total once; each parent receives one partial per child
 * and sends the total once per child. */
static int tree_rank_at(int t, int n, int pos) {
  return t == 0 ? pos : n - 1 - pos;
}

int orc_allreduce_tree(int n, size_t count, int dt, const void* const* in, void* const* out,
                       uint64_t* sent, uint64_t* recv) {
  if (n < 1 || n > 64) return ORC_EINVAL;
  size_t e = elem_size(dt);
  size_t half[3];
  orc_chunk_plan(2, count, dt, half);
  /* part[p]: the partial of the node at heap position p */
  void** part = (void**)calloc((size_t)n, sizeof(void*));
  if (!part) return ORC_ENOMEM;
  int rc = ORC_OK;
  for (int p = 0; p < n; ++p) {
    part[p] = malloc(count * 4 + 4);
    if (!part[p]) { rc = ORC_ENOMEM; goto done; }
  }
  for (int t = 0; t < 2; ++t) {
    const size_t lo = half[t], len = half[t + 1] - half[t];
    /* reduce up: children sit at larger positions, so descending positions
     * finish every child before its parent */
    for (int p = n - 1; p >= 0; --p) {
      const int r = tree_rank_at(t, n, p);
      acc_load(dt, in[r], lo, len, part[p]);
      for (int child = 2 * p + 1; child <= 2 * p + 2; ++child) {
        if (child >= n) continue;
        tally(sent, tree_rank_at(t, n, child), len * e);
        tally(recv, r, len * e);
        if (dt == ORC_INT32)
          for (size_t i = 0; i < len; ++i) ((uint32_t*)part[p])[i] += ((uint32_t*)part[child])[i];
        else
          for (size_t i = 0; i < len; ++i) ((float*)part[p])[i] = ((float*)part[p])[i] + ((float*)part[child])[i];
      }
    }
    /* broadcast down: the root's rounded total, forwarded unchanged */
    acc_store(dt, part[0], out[tree_rank_at(t, n, 0)], lo, len);
    for (int p = 1; p < n; ++p) {
      const int r = tree_rank_at(t, n, p), parent = tree_rank_at(t, n, (p - 1) / 2);
      memcpy((char*)out[r] + lo * e, (const char*)out[parent] + lo * e, len * e);
      tally(sent, parent, len * e);
      tally(recv, r, len * e);
    }
  }
done:
  for (int p = 0; p < n; ++p) free(part[p]);
  free(part);
  return rc;
}
