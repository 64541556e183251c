// Launch interface between the host API (api.cu) and the kernels (engine.cu).
#pragma once

#include <cuda.h>  // CUtensorMap (the type only; maps are encoded through the runtime)
#include <cuda_runtime.h>
#include <stdint.h>

#include "coll_internal.h"

namespace coll {

struct RankPtrs {
  const char *in[COLL_MAX_RANKS];
  char *out[COLL_MAX_RANKS];
};

struct ZcArgs {
  RankPtrs ptr;
  const coll_job_t *jobs;
  const coll_ref_t *refs;
  const coll_tile_t *tiles;
  const coll_btile_t *btiles;  // bulk kernel: the same tiles with their references inlined
  uint32_t ntiles;
  uint32_t n_epochs;
  int32_t in_pool;
  int32_t pad;
  int64_t in_stride, out_stride;
  coll_dev_status_t *st;  // bulk kernel: timeout reporting
  uint64_t spin_ns;       // bulk kernel: bound on every mbarrier wait
  uint32_t slot_bytes;    // bulk kernel: bytes per staged piece
  uint32_t stages;        // bulk kernel: ring depth
  uint32_t maxsrc;        // bulk kernel: slots per stage
  uint32_t tree;          // 1: pairwise (tree) summation order within groups of 8
  uint64_t static_tiles;  // bulk kernel: tiles dealt round-robin; the rest are claimed
  uint32_t dyn_tail;      // bulk kernel: claim the last fifth of the tiles dynamically,
                          // 1: two at a time, 2: in guided sizes (long runs only)
  uint32_t pad2;
};

struct EngArgs {
  RankPtrs ptr;                        // fused producer: ptr.in[r] is the GEMV vector x_r
  const char *wt[COLL_MAX_RANKS];      // fused producer: W_r transposed, [k][in_len[r]] bf16
  int64_t wt_stride[COLL_MAX_RANKS];   // bytes per row of wt[r]
  uint32_t gemv_k;                     // 0: stage loads its payload; k: stage computes W_r x_r
  uint32_t gemv_pitch;                 // fused producer: bytes per staged weight row (the
                                       // unit's bytes: its columns x 2)
  uint32_t gemv_slots;                 // fused producer: slots of the weight ring
  const coll_unit_t *units;
  const coll_item_t *sitems;
  const coll_item_t *citems;
  const coll_warp_t *warps;
  const coll_ref_t *refs;
  char *xbuf;
  uint64_t xpar;
  unsigned long long *pflag;  // [2][n_pflag] {epoch:16, tag B:16, tag A:32}
  uint32_t *cflag;            // [n_cflag]
  const coll_item_t *pitems;  // two-shot pull: pull items (unit, consumer slot)
  char *rbuf;                 // two-shot pull: reduced pieces, [parity] x rpar bytes
  uint64_t rpar;
  uint32_t *rflag;            // two-shot pull: [2][n_units] epoch of each reduced piece
  uint32_t *dflag;            // two-shot pull: epoch each consumer has pulled
  uint32_t n_units;
  coll_dev_status_t *st;
  uint64_t *stamps;           // [stamp_cap + 1] or null
  uint32_t *dbg;              // [n_units] handshake words of the SPEC_PAUSE injection
  uint32_t *rank_done;        // [R] chained epochs: consume completions per rank
  int32_t chain;
  uint32_t stamp_cap;
  uint32_t stamp_phases;  // 1: four stamps per epoch (start, notified, data ready, end)
  uint32_t n_pflag;
  uint32_t nwarps;
  int32_t n_epochs;
  int32_t in_pool;
  uint32_t epoch_base;  // epochs already run by this plan; epoch i of this run is base+i+1
  int64_t in_stride, out_stride;
  int32_t protocol;
  int32_t spec_check;
  uint64_t spin_ns;
  uint64_t inject_flags;
  uint64_t inject_seed;
  int32_t inject_rank;
  uint32_t inject_prob_ppm;
  uint64_t inject_max_ns;
  uint64_t inject_start_ns;
  uint64_t inject_pause_ns;
  int32_t R;
  uint32_t single_items;  // 1: every warp has one stage item and one consume item
  uint32_t spec_delay_ns; // speculative protocol: wait before the first speculative loads
  uint32_t spec_adapt;    // 1: each warp adapts that wait to its own failed first attempts
};

// Fused producer: one 2-D tensor map per rank over W_r ([k rows][in_len[r] bf16 columns],
// box of 256 columns x 64 rows), passed by value as a kernel parameter.
struct GemvMaps {
  CUtensorMap m[COLL_MAX_RANKS];
};
struct NoMaps {
  uint32_t unused;
};

// Zero-copy: one ordinary launch over all tiles of all epochs.
cudaError_t launch_zero_copy(int op, int dtype, int oneshot_reuse, const ZcArgs &a, int ctas,
                             cudaStream_t s);

// Zero-copy, bulk (TMA) ring: one launch of `ctas` persistent CTAs (one per SM).
cudaError_t launch_bulk(int op, int dtype, const ZcArgs &a, int ctas, cudaStream_t s);
uint32_t bulk_smem_bytes(uint32_t stages, uint32_t maxsrc, uint32_t slot_bytes);

// Staged Stage/Notify/Consume engine: one cooperative launch of nwarps one-warp CTAs (twelve
// warps each for the fused producer, which needs `maps`; null otherwise).
cudaError_t launch_engine(int op, int dtype, const EngArgs &a, const GemvMaps *maps,
                          cudaStream_t s);

// Flag ping-pong probe between block 0 and block `peer` (cooperative launch).
cudaError_t launch_probe_rtt(unsigned long long *flags, uint32_t iters, uint32_t peer,
                             unsigned long long *out, uint64_t limit, cudaStream_t s);

// How many one-warp engine CTAs can be co-resident on the current device.
cudaError_t engine_max_coresident(int op, int dtype, int protocol, int datapath, int *max_ctas);

// Slots of the fused producer's weight ring for staged rows of `pitch` bytes.
uint32_t gemv_ring_slots(uint32_t pitch);

// How many fused-producer engine CTAs (twelve warps, a 192 KiB weight ring) can be co-resident.
cudaError_t engine_gemv_max_coresident(bool pull, int *max_ctas);

}  // namespace coll
