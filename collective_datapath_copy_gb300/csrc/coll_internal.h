// Internal plan tables shared by the host plan compiler (plan.cpp) and the device code
// (engine.cu). Not part of the C ABI.
#pragma once

#include <stdint.h>

#include "coll.h"

#define COLL_MAX_RANKS 64
#define COLL_MAX_ELEMS (1ull << 48)  // elements in one rank's buffer
#define COLL_MAX_FANIN 256   // producers of one name
#define COLL_MAX_FANOUT 256  // consumers of one name
#define COLL_WARP_VEC 32     // lanes per warp, one 16-byte vector each per step
#define COLL_BULK_MAX_SRC 8  // bulk (TMA) zero-copy path: producers per job
#define COLL_BULK_MAX_DST 8  // bulk (TMA) zero-copy path: consumers per job

// (rank, byte offset) of one segment inside that rank's buffer.
struct coll_ref_t {
  uint32_t rank;
  uint32_t pad;
  uint64_t off;
};

// Zero-copy datapath: a job moves one name's bytes from nsrc producer segments (summed in
// the stored order, which is (rank, offset) ascending) into ndst consumer segments.
struct coll_job_t {
  uint32_t src0, nsrc;  // refs[src0 .. src0+nsrc)
  uint32_t dst0, ndst;  // refs[dst0 .. dst0+ndst)
};

// A tile: bytes [start, start+nbytes) of every segment of one job.
struct coll_tile_t {
  uint32_t job;
  uint32_t nbytes;
  uint64_t start;
};

// Staged datapath: a synchronisation unit is one piece (<= unit_bytes) of one name.
// Producer slot j stages its piece into the exchange buffer at xoff + j * nbytes of the
// current parity and notifies pflag[parity][pflag0 + j]; a consumer waits for / validates
// those flags and reduces or copies the pieces into its output segment(s).
#define COLL_UNIT_REUSE_WAIT 1u  // stagers must wait for consumers' done flags (dual/spec)
#define COLL_UNIT_DONE_FLAGS 2u  // consumers write done flags
#define COLL_UNIT_PULL 4u        // two-shot pull: the owner writes the reduced piece to rbuf
struct coll_unit_t {
  uint64_t start;   // byte offset inside the name's segments
  uint64_t xoff;    // byte offset of slot 0 inside one parity of the exchange buffer
  uint32_t nbytes;  // multiple of 16
  uint32_t src0, nsrc;
  uint32_t dst0, ndst;
  uint32_t pflag0;  // producer flag base (per parity)
  uint32_t cflag0;  // consumer done-flag base
  uint32_t ncflag;  // number of done flags (ndst for oneshot/copy, 1 for twoshot)
  uint32_t flags;   // COLL_UNIT_*
  uint32_t dflag0;  // two-shot pull: base of the ndst pulled flags (consumer i read rbuf)
  uint64_t roff;    // two-shot pull: offset of the reduced piece in one parity of rbuf
};

// Zero-copy bulk ring: one tile with its sources and destinations inlined (rank in the
// top 8 bits, segment byte offset below), so that resolving a tile is one memory round trip.
#define COLL_BULK_REF(rank, off) (((uint64_t)(rank) << 56) | (uint64_t)(off))
struct coll_btile_t {
  uint64_t start;   // byte offset inside the job's segments
  uint32_t nbytes;
  uint16_t nsrc, ndst;
  uint64_t ref[COLL_BULK_MAX_SRC + COLL_BULK_MAX_DST];  // sources, then destinations
};

#define COLL_SLOT_ALL 0xFFFFFFFFu
struct coll_item_t {
  uint32_t unit;
  uint32_t slot;  // producer slot (stage) / consumer slot (consume) / ALL (twoshot owner)
};

struct coll_warp_t {
  uint32_t rank;
  uint32_t s0, s1;  // stage items
  uint32_t c0, c1;  // consume items
  uint32_t rank_warps;  // warps of this rank (chained epochs count them)
  uint32_t p0, p1;      // pull items (two-shot pull)
};

// Device status block of a plan (zeroed at plan time and by coll_reset).
struct coll_dev_status_t {
  int32_t status;
  int32_t fail_rank;
  int32_t fail_unit;
  int32_t fail_where;
  uint64_t fail_epoch;
  uint32_t abort;
  uint32_t pad;
  unsigned long long spec_checks;
  unsigned long long spec_retries;
  uint32_t tail_claim;  // zero-copy bulk ring: tiles of the dynamic tail claimed so far
  uint32_t tail_done;   // ... and CTAs finished (the last one resets both to zero)
};

// Host-side compiled plan (no device pointers); built by coll_compile().
#ifdef __cplusplus
#include <vector>
struct coll_compiled {
  int R = 0, op = 0, dtype = 0, esize = 0;
  coll_config_t cfg{};
  std::vector<uint64_t> in_bytes, out_bytes;  // per-rank buffer sizes in bytes
  std::vector<uint8_t> in_used, out_used;     // rank has segments
  std::vector<coll_ref_t> refs;
  std::vector<coll_job_t> jobs;
  std::vector<coll_tile_t> tiles;
  std::vector<coll_btile_t> btiles;  // bulk ring plans: tiles with inlined references
  std::vector<coll_unit_t> units;
  std::vector<coll_item_t> sitems, citems, pitems;
  std::vector<coll_warp_t> warps;
  bool zc_keep = false;       // zero-copy: inputs are re-read (one-shot sums with several
                              // consumers per name): keep them cacheable
  bool bulk = false;          // zero-copy tiles sized for the bulk (TMA) kernel
  uint32_t bulk_slot = 0;     // bytes of one staged piece (= tile size)
  uint32_t bulk_maxsrc = 0;   // slots per stage
  uint32_t bulk_stages = 0;   // stages in the shared-memory ring
  uint32_t bulk_tail = 0;     // claim the last tiles dynamically: 1 two at a time, 2 in
                              // guided sizes (see bulk.cu)
  uint64_t xpar_bytes = 0;  // exchange bytes per parity
  uint64_t rpar_bytes = 0;  // two-shot pull: reduced-piece bytes per parity
  uint32_t n_pflag = 0, n_cflag = 0, n_dflag = 0;
  uint64_t n_names = 0, min_bytes = 0;
};

int coll_compile(int R, int op, int dtype, const coll_seg_t *in_segs, size_t n_in,
                 const uint64_t *in_len, const coll_seg_t *out_segs, size_t n_out,
                 const uint64_t *out_len, const coll_config_t *cfg, int max_warps,
                 int num_sms, coll_compiled *out);
// Engine warps that may be co-resident when no device can be asked (host-only compile).
inline int coll_default_max_warps() { return 1024; }
inline int coll_default_num_sms() { return 152; }
void coll_fill_info(const coll_compiled &c, coll_plan_info_t *info);
#endif
