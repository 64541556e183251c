/*
 * coll.h — C ABI of the collective datapath (libcoll.so), GB300 / sm_103a.
 *
 * A collective is stated as a NAMING: each rank's input buffer and output buffer are cut
 * into segments, every segment carries a name, and an operation (copy or sum) says what an
 * output segment receives from the input segments that carry its name.
 *   Source: Purlin article, "The Purlin PDF describes a three-layer design" (collectives
 *   as a naming of an input and an output layout plus copy or reduction; a shared
 *   Stage / Notify / And Consume orchestration; an Atom datapath with copy and reduce).
 * The R ranks are emulated on one GPU: rank r is the buffer pair (in[r], out[r]) plus the
 * group of warps that produces rank r's data and consumes rank r's outputs.
 *
 * Semantics of one epoch (independent of protocol, timing and retries):
 *   copy: an output segment receives the bytes of the single input segment with its name.
 *   sum : an output segment receives, per element, the binary32 chain
 *         acc = x_0; acc = acc + x_k (k = 1..n-1, round to nearest even, no FMA), over the
 *         input segments with its name ordered by (rank, offset) ascending; bf16 outputs
 *         are rounded once from acc, to nearest even. Results are bit-exact.
 *   Output elements that no segment names are not written.
 *
 * Threading: the library is thread-safe across plans; a plan allows one run in flight
 * (a second coll_run on another stream before the first finished is undefined).
 * All pointers passed to coll_run are device pointers of the current device.
 */
#ifndef COLL_H
#define COLL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ codes */
#define COLL_OK 0
#define COLL_EINVAL (-1)    /* bad R (1..64), op, dtype, rank, count 0, config value   */
#define COLL_ENAME (-2)     /* a consumed name has no producer, or copy with >1        */
#define COLL_ELEN (-3)      /* segments with one name have different counts            */
#define COLL_EBOUNDS (-4)   /* offset+count beyond the rank's buffer length            */
#define COLL_EOVERLAP (-5)  /* output segments of one rank overlap; or (coll_run)
                               output memory overlaps input or another output         */
#define COLL_EALIGN (-6)    /* staged (non zero-copy) plans need 16-byte-aligned segment
                               byte offsets/sizes; coll_run needs 16-byte-aligned bases */
#define COLL_ECUDA (-7)     /* a CUDA runtime call failed (launch, memory)              */
#define COLL_ETIMEDOUT (-8) /* async: a bounded device wait expired; kernel returned    */
#define COLL_EDEVICE (-9)   /* async: the device reported an inconsistent state         */
#define COLL_ENOMEM (-10)   /* host or device allocation failed                         */
#define COLL_ETOOBIG (-11)  /* coll_allreduce_static: the request needs more than its fixed
                               scratch array or more warps than can be co-resident       */

/* ------------------------------------------------------------------ enums */
#define COLL_OP_COPY 0
#define COLL_OP_SUM 1

#define COLL_BF16 0  /* 2-byte elements; sum accumulates in binary32          */
#define COLL_F32 1   /* 4-byte elements                                       */
#define COLL_BYTES 2 /* 1-byte elements; copy only                            */

/* Stage/Notify/Consume protocols for staged plans (zero_copy == 0).
 * Source: SiFAR review, "What carries the argument" and abstract: oneshot with a top and a
 * bottom barrier; dual buffering (epoch parity) removes the bottom barrier; speculative
 * reduction starts the transfer before the top barrier and validates with a reduced flag,
 * retrying on mismatch. */
#define COLL_PROTO_BARRIER 0
#define COLL_PROTO_DUAL 1
#define COLL_PROTO_SPEC 2
/* Lamport-style tagged data (the pages' push-based baseline, SiFAR review, Fig. 20): dual
 * buffers whose 8-byte words each carry 4 payload bytes and the epoch; a consumer polls the
 * words themselves until every tag shows its epoch. 8-byte single-copy atomicity validates
 * every word: no flags, no fence, no hash; twice the exchange bytes. */
#define COLL_PROTO_LL 3

/* Datapaths for sum. Source: SiFAR review, Fig. 5 (oneshot: every consumer reduces the
 * whole payload from every producer) and Fig. 6 (twoshot: each part is reduced once, by an
 * owner, and then delivered to every consumer). TWOSHOT: the owner writes the reduced part
 * to every consumer (push). TWOSHOT_PULL (staged plans only, not with COLL_PROTO_LL): the
 * owner writes it to a second exchange buffer and notifies; every consumer waits for that
 * flag and copies the part into its output (the all-gather pull of the pages), then signals
 * that it has read it; the owner waits for those signals before it overwrites the buffer
 * (the two-shot bottom barrier). Same result bits as ONESHOT and TWOSHOT. */
#define COLL_DP_ONESHOT 0
#define COLL_DP_TWOSHOT 1
#define COLL_DP_TWOSHOT_PULL 2

/* Summation order of sums (zero-copy plans). RANK is the fixed rank order and is
 * bit-exact; TREE adds each group of up to 8 producers pairwise ((x0+x1)+(x2+x3))+...,
 * groups in order: a different rounding order, accurate to the first-order bound of any
 * summation order, (n-1) * 2^-24 * sum|x|, plus the output rounding. */
#define COLL_ORDER_RANK 0
#define COLL_ORDER_TREE 1

/* Speculative validation rules (COLL_PROTO_SPEC). A producer publishes one 64-bit flag word
 * per piece, {epoch mod 2^16, tag B mod 2^16, tag A}: two independent content hashes of the
 * piece (32 and 16 bits kept) with the epoch folded in. A stale or torn read passes the
 * tagged checks only if both collide (about 2^-48 per stale read). */
#define COLL_SPEC_TAGGED 0  /* flag epochs AND the content tags must match (sound)      */
#define COLL_SPEC_LITERAL 1 /* only sum of flag epochs == n * epoch (the pages' rule);
                               unsound under reordering, kept as an ablation            */
#define COLL_SPEC_TAGGED_RELAXED 2 /* content tags only: notify without a release fence,
                                      validate by re-hashing and re-load until the tags
                                      match (bounded); no reliance on memory ordering   */

/* Host-driven fault / timing injection (never a GPU fault; every wait stays bounded). */
#define COLL_INJECT_SKIP_NOTIFY (1ull << 0) /* rank inject_rank never notifies          */
#define COLL_INJECT_STAGGER (1ull << 1)     /* random per-epoch rank delays + start skew */
#define COLL_INJECT_SPEC_PAUSE (1ull << 2)  /* adversarial interleaving: consumers of
                                               inject_rank load speculatively, signal,
                                               pause inject_pause_ns, then read the flags;
                                               rank inject_rank+1 stages each piece only
                                               after that signal (waiting at most
                                               inject_max_ns): payload read, then peer
                                               write + flag, then flag read              */

typedef struct coll_plan_s *coll_plan_t;

/* One segment: elements [offset, offset+count) of rank `rank`'s buffer carry `name`. */
typedef struct {
  int32_t rank;
  int32_t reserved; /* must be 0 */
  uint64_t offset;  /* elements */
  uint64_t count;   /* elements, > 0 */
  uint64_t name;
} coll_seg_t;

typedef struct {
  int32_t protocol;       /* COLL_PROTO_*; staged plans only                          */
  int32_t datapath;       /* COLL_DP_*; sum only                                      */
  int32_t zero_copy;      /* 1: consumers read the inputs directly, one kernel per
                             coll_run, no exchange buffers or flags (the kernel launch
                             is the barrier). 0: staged Stage/Notify/Consume engine.   */
  int32_t spec_check;     /* COLL_SPEC_*                                              */
  int32_t unit_bytes;     /* staged: bytes per synchronisation unit (one warp's piece):
                             0 (= 512) or a multiple of 16 from 64 to 512               */
  int32_t warps_per_rank; /* staged: warps per emulated rank; 0 = one per unit        */
  int32_t ctas;           /* zero-copy: CTAs (8 warps each) in the grid; 0 = 3 x SMs  */
  int32_t tile_bytes;     /* zero-copy: bytes per warp tile, multiple of 16; 0 = auto
                             (512 B .. 32 KiB, about four tiles per resident warp)     */
  uint64_t tma_min_bytes; /* zero-copy plans whose jobs move at least this many bytes,
                             with 16-byte-aligned segments and <= 8 producers and
                             consumers per job, use the bulk-copy (TMA) ring kernel;
                             0 = 4 MiB; UINT64_MAX = never                             */
  uint64_t spin_limit_ns; /* bound on every device wait; 0 = 2e9 (2 s)                  */
  uint32_t record_stamps; /* staged: 1 = one %globaltimer stamp per epoch (capacity
                             stamp_capacity epochs; later epochs are not stamped);
                             2 = four per epoch (start, notified, data ready, end) of
                             the first warp                                            */
  uint32_t stamp_capacity;
  uint64_t inject_flags;  /* COLL_INJECT_*                                            */
  uint64_t inject_seed;
  int32_t inject_rank;
  uint32_t inject_prob_ppm; /* STAGGER: probability per epoch, parts per million      */
  uint64_t inject_max_ns;   /* STAGGER: max delay; SPEC_PAUSE: producer's bounded wait */
  uint64_t inject_start_ns; /* STAGGER: rank r starts r * inject_start_ns late          */
  uint64_t inject_pause_ns; /* SPEC_PAUSE: consumer pause                              */
  int32_t chain;            /* staged: 1 = rank r stages epoch e+1 only after every one of
                               its consume items of epoch e is done (a dependent chain, as
                               when the next layer needs the whole all-reduce output);
                               0 = back-to-back independent epochs                       */
  int32_t spec_delay_ns;    /* COLL_PROTO_SPEC: ns a consumer waits after its own notify
                               before its first speculative loads (loads issued at once
                               mostly race the peers' stores of the same epoch and are
                               retried): -1 = the check's default: for
                               COLL_SPEC_TAGGED_RELAXED a window per warp that starts at
                               200 ns, grows by 2 ns after a first attempt that failed
                               and passed at the first reload (a race) and shrinks by
                               1/8 ns after one that passed (about one in seventeen then
                               fails), no window for the other checks; 0..100000 = that
                               many ns, fixed                                            */
  int32_t reduce_order;     /* COLL_ORDER_*; zero-copy plans only                      */
  int32_t reserved3;        /* must be 0                                                */
} coll_config_t;

typedef struct {
  uint64_t n_names;      /* consumed names                                           */
  uint64_t n_jobs;       /* zero-copy jobs (a job = sources -> destinations)          */
  uint64_t n_tiles;      /* zero-copy tiles                                           */
  uint64_t n_units;      /* staged synchronisation units                              */
  uint64_t n_warps;      /* staged engine warps (= CTAs of 32 threads)                */
  uint64_t min_bytes;    /* algorithmic bytes per epoch: every input byte a named output
                            depends on read once + every named output byte written once */
  uint64_t xbuf_bytes;   /* staged exchange buffers (both parities)                   */
  uint64_t flag_bytes;   /* staged flag words                                         */
  uint64_t bulk_tile_bytes; /* zero-copy: bytes per tile of the bulk (TMA) ring kernel the
                               plan was compiled for; 0 = the warp kernel               */
} coll_plan_info_t;

typedef struct {
  int32_t status;        /* COLL_OK, COLL_ETIMEDOUT or COLL_EDEVICE of the last run    */
  int32_t fail_rank;     /* timeout: rank of the warp that gave up (-1 if none)        */
  int32_t fail_unit;     /* timeout: unit it waited on                                 */
  int32_t fail_where;    /* 1 stage reuse wait, 2 consume wait, 3 retry wait, 4 output
                            completion wait                                           */
  uint64_t fail_epoch;   /* timeout: epoch number it waited for                        */
  uint64_t epochs;       /* epochs completed by this plan, all runs                    */
  uint64_t spec_checks;  /* speculative validations (units x epochs)                   */
  uint64_t spec_retries; /* validations that failed and were redone after a wait       */
} coll_stats_t;

/* Fill *cfg with defaults (spec protocol with the fence-free tagged check and its default
 * speculation delay, oneshot, staged).
 * Source: SiFAR review, "What carries the argument" (speculative reduction over dual
 * buffers is the protocol the review's All-Reduce is built on). */
int coll_config_default(coll_config_t *cfg);

/* Validate a naming and compile it into a plan: host work tables, device tables,
 * exchange buffers (x2 parities) and zeroed flags for staged plans.
 * Source: Purlin article, "The Purlin PDF describes a three-layer design": the top layer
 * states a collective as a naming of an input and an output layout plus copy or reduction,
 * and SNAC derives the coordination from that statement; here the plan compiler derives
 * which warp stages, notifies and consumes each piece, and which flags each consumer reads.
 * R: 1..64 ranks. in_len/out_len: R buffer lengths in elements, each at most 2^48
 * (COLL_EBOUNDS beyond). cfg may be NULL (defaults).
 * Ownership: the plan owns everything it allocates; coll_free releases it. The segment
 * arrays are copied and may be freed after the call.
 * Errors (synchronous, nothing allocated): COLL_EINVAL, COLL_EBOUNDS, COLL_ELEN,
 * COLL_ENAME, COLL_EOVERLAP (in that order of precedence), COLL_EALIGN, COLL_ENOMEM,
 * COLL_ECUDA. */
int coll_plan(coll_plan_t *out, int R, int op, int dtype, const coll_seg_t *in_segs,
              size_t n_in, const uint64_t *in_len, const coll_seg_t *out_segs, size_t n_out,
              const uint64_t *out_len, const coll_config_t *cfg);

/* The host half of coll_plan only: same checks and codes, no device call (usable on a
 * machine without a GPU). info may be NULL.
 * Source: as coll_plan (Purlin article, "three-layer design": the naming layer). */
int coll_validate(int R, int op, int dtype, const coll_seg_t *in_segs, size_t n_in,
                  const uint64_t *in_len, const coll_seg_t *out_segs, size_t n_out,
                  const uint64_t *out_len, const coll_config_t *cfg,
                  coll_plan_info_t *info);

/* Sizes of a compiled plan and its minimal (algorithmic) bytes per epoch. No counterpart
 * on the pages; the minimal bytes are the denominator of the bandwidth figures. */
int coll_plan_info(coll_plan_t p, coll_plan_info_t *info);

/* Run n_epochs epochs of the plan on `stream` (a cudaStream_t; NULL = legacy default).
 * Source: Purlin article, "three-layer design" (Stage, Notify, And Consume orchestrates the
 * Atom datapath's copy and reduce); SiFAR review, "What carries the argument" and Figs. 5
 * and 6 (the protocols and the oneshot / twoshot datapaths a staged plan runs).
 * in/out: host arrays of R device pointers. Epoch i (0-based) reads
 * in[r] + (i % in_pool) * in_epoch_stride bytes and writes out[r] + i * out_epoch_stride
 * bytes (stride 0 overwrites). A rank with no segments may pass NULL.
 * Staged plans run one cooperative persistent launch for all epochs; zero-copy plans run
 * one ordinary launch. Returns after enqueueing; device-side failures are reported by
 * coll_status. Runs may be captured into a CUDA graph (the plan's tables are fixed; the
 * pointers and strides given here are baked into the captured launch). Once a staged plan
 * has been captured, each of its runs, the captured one with every replay included, first
 * clears the plan's flags on the stream and counts its epochs from 1. A plan still runs one
 * run at a time: replays and direct runs of it must not overlap.
 * Synchronous errors: COLL_EINVAL (n_epochs < 1, in_pool < 1, NULL pointer
 * for a rank that has segments), COLL_EALIGN, COLL_EOVERLAP, COLL_ECUDA. Buffers must stay
 * live and unmodified until the stream has passed the run. */
int coll_run(coll_plan_t p, void *const *in, void *const *out, int n_epochs,
             int64_t in_epoch_stride, int in_pool, int64_t out_epoch_stride, void *stream);

/* Fused producer (staged bf16 plans): like coll_run, but each rank's payload is computed
 * inside the engine's stage step instead of read from memory — the layer that precedes the
 * collective fused into its persistent loop (SiFAR review, Summary: the All-Reduces run
 * inside megakernels, after each layer's computation). At epoch i rank r's input buffer
 * (in_len[r] bf16 elements, the buffer the naming refers to) is y_r = W_r x_r(i): wt[r] is
 * W_r given transposed, k rows of in_len[r] bf16 (row stride in_len[r] elements), and
 * x_r(i) = x[r] + (i % x_pool) * x_epoch_stride bytes holds k bf16. Element j of y_r is the
 * plain dot product: the k products wt[r][i][j] * x_r(i)[i], each rounded to binary32, added
 * in row order i = 0..k-1 from the first product (round to nearest even, no fused
 * multiply-add), then rounded once to bf16. Results are bit-exact. Each engine CTA runs
 * eight warps in this mode (four compute, two streaming the weight rows and x into shared
 * memory by tensor and bulk copies), one CTA per SM, and computes one unit of the plan
 * (coll_config_t.unit_bytes: units of 432 bytes spread an 8 KiB payload of 8 ranks over 152
 * SMs instead of 128); without chained epochs the next piece
 * is computed while the current one is exchanged. k must be a multiple of 16, at most
 * 8192; in_len[r], wt[r], x[r] and the strides must give 16-byte alignment, and in_len[r]
 * must be below 2^32. The tensor maps of W_r are encoded on the host at the first run with
 * these matrices (and again when wt or k change).
 * Errors as coll_run, plus COLL_EINVAL for a zero-copy, tagged-data or non-bf16 plan, a k
 * outside those limits, or a plan with more warps than SMs can hold fused CTAs at once. */
int coll_run_gemv(coll_plan_t p, const void *const *wt, void *const *x, int k, void *const *out,
                  int n_epochs, int64_t x_epoch_stride, int x_pool, int64_t out_epoch_stride,
                  void *stream);

/* Wait for the plan's last run and report its status and counters. Returns the run's
 * status (COLL_OK, COLL_ETIMEDOUT, COLL_EDEVICE) or COLL_ECUDA. st may be NULL.
 * Source: SiFAR review, Referee Report, major comment 1 and Figs. 23-25 (validations that
 * fail are retried, and the mis-speculation rate is reported: spec_checks, spec_retries);
 * "What would settle it" (a wait that never ends is the failure to detect: a bounded wait
 * ends the run with COLL_ETIMEDOUT and fail_* say where). */
int coll_status(coll_plan_t p, coll_stats_t *st);

/* Copy up to n per-epoch %globaltimer stamps (ns) of the last run into host memory;
 * returns the number copied (synchronises on the last run).
 * Source: SiFAR review, Fig. 15 and Referee Report minor comment 4 (latency per payload /
 * TP cell): the stamps give the per-epoch latency distribution of a run. */
int64_t coll_stamps(coll_plan_t p, uint64_t *host, int64_t n);

/* Measurement probe (not part of the collective; SiFAR review, "If this is right": once
 * GPUs are in lockstep, the top barrier costs a flag exchange): ping-pong one flag `iters` times
 * between one thread of block 0 and one thread of block `peer_block` of a cooperative
 * launch with peer_block+1 one-warp blocks, and report the total ns (%globaltimer) and the
 * two SM ids. This is the round trip that bounds a flag handshake between two emulated
 * ranks. Synchronous; allocates and frees 1 KiB. COLL_ETIMEDOUT if a wait exceeded 1 s. */
int coll_probe_flag_rtt(int peer_block, int iters, uint64_t *ns_total, int *sm_a, int *sm_b);

/* Wait for the last run, then re-zero flags, counters and the epoch counter. After a run
 * that reported COLL_ETIMEDOUT the plan's flags are inconsistent: call this before the next
 * coll_run on the plan. No counterpart on the pages (the flags of the SNAC layer restart). */
int coll_reset(coll_plan_t p);

/* Wait for the last run and release everything the plan owns. NULL is a no-op.
 * Source: Purlin article, "three-layer design" (the plan holds the SNAC layer's exchange
 * buffers and flags for one naming; freeing it ends that naming's coordination). */
int coll_free(coll_plan_t p);

/* All-reduce (sum) that allocates nothing. The pages have no counterpart: this exists for
 * callers that cannot allocate device memory when they need the collective — a serving
 * process that reserved nearly all HBM up front for weights and the KV cache (a late
 * cudaMalloc fails or fragments that reservation), or a latency-critical loop where a
 * cudaMalloc/cudaFree pair would add an implicit device synchronisation. It calls no
 * allocating routine.
 * Same result as coll_plan/coll_run for an all-reduce naming (every rank's whole buffer is
 * one name) with the dual-buffer protocol: out[r] = the rank-order binary32 sum of all R
 * inputs, rounded once to bf16 for COLL_BF16. in/out: host arrays of R device pointers,
 * 16-byte aligned, count elements each; epochs, pool and strides as in coll_run; inputs
 * and outputs must not overlap. status: optional device int32 the kernel sets to
 * COLL_ETIMEDOUT if a bounded wait expires (cleared by the call; NULL = not reported).
 * Scratch: a fixed 4 MiB device array held by every GPU that loads the library until the
 * process exits; it holds 2 x R x ceil(count*size/512) pieces of 512 bytes plus flags, so
 * R x count x element size up to about 2 MiB fits. Larger requests (or more warps than can
 * be co-resident), including any count whose byte size exceeds the array, return
 * COLL_ETOOBIG. The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture. Every call shares the array and clears its flags on `stream`
 * first; calls that can overlap on the GPU (other streams, unordered) race on it.
 * Errors: COLL_EINVAL, COLL_EALIGN, COLL_ETOOBIG, COLL_ECUDA (synchronous). */
int coll_allreduce_static(int R, int dtype, void *const *in, void *const *out, uint64_t count,
                          int n_epochs, int64_t in_epoch_stride, int in_pool,
                          int64_t out_epoch_stride, int32_t *status, void *stream);

/* Static string for a code. No counterpart on the pages. */
const char *coll_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* COLL_H */
