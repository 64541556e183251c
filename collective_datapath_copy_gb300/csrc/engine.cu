// Kernels of the collective datapath for sm_103a.
//
// zc_kernel     — zero-copy datapath: every consumer reads the producers' input buffers
//                 directly; the kernel launch itself orders producers before consumers.
// engine_kernel — the staged Stage / Notify / Consume engine: a persistent cooperative
//                 launch in which one warp per CTA plays part of one emulated rank and
//                 loops over epochs, synchronising with the other ranks' warps only
//                 through epoch flags in global memory.
//
// Sources: Purlin article, "The Purlin PDF describes a three-layer design" (naming,
// SNAC = Stage / Notify / And Consume, Atom copy/reduce); SiFAR review, "What carries the
// argument", abstract and Figs. 5, 6, 14 (oneshot and twoshot, top and bottom barriers,
// dual buffering, speculative reduction validated by a reduced flag with retry).
#include <cuda_runtime.h>
#include <stdint.h>

#include "atom.cuh"
#include "engine.cuh"
#include "tma.cuh"

namespace coll {

namespace {

constexpr unsigned FULL = 0xFFFFFFFFu;

// ============================================================== zero-copy datapath

// KIND: 0 copy (bytes), 1 sum of bf16, 2 sum of f32.
// KEEP: inputs are read again by other tiles (oneshot) -> keep them cacheable; otherwise
//       every input byte is read once and streamed.
template <int KIND, bool KEEP>
__device__ __forceinline__ uint4 zc_load(const char *p) {
  if constexpr (KEEP) return ld_nc_v4(p); else return ld_cs_v4(p);
}

// One warp per tile. Lane k holds the pointer of producer k and of consumer k for the
// tile (up to 32 each); the vector loops fetch them with shuffles. Tiles with more than 32
// producers or consumers, or with an address not 16-byte aligned, take the element-wise
// path (same arithmetic, same order). The kernel is launched as a programmatic dependent of
// the previous kernel in its stream: each CTA lets the next kernel start at once (which waits
// for this one before it touches caller buffers), and each warp reads its first tile's
// record, the plan's, before it waits for the previous kernel (griddep_wait) and touches
// the caller's buffers.
template <int KIND, bool KEEP, bool TREE>
__global__ void __launch_bounds__(256, TREE ? 2 : 3) zc_kernel(const ZcArgs a) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint64_t gw = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint64_t nw = ((uint64_t)gridDim.x * blockDim.x) >> 5;
  const uint64_t total = (uint64_t)a.ntiles * a.n_epochs;
  constexpr uint64_t kOffMask = (1ull << 56) - 1u;
  griddep_launch();
  bool waited = false;  // the previous kernel in the stream has completed
  for (uint64_t t = gw; t < total; t += nw) {
    const uint32_t e = (uint32_t)(t / a.ntiles);
    const uint32_t ti = (uint32_t)(t - (uint64_t)e * a.ntiles);
    // The tile's segments: from its inline record when the plan has one (one memory round
    // trip: lanes 0..17 read the record's 8-byte words), else through tile -> job -> refs.
    const uint64_t *rec = a.btiles ? reinterpret_cast<const uint64_t *>(a.btiles + ti) : nullptr;
    uint64_t start, word = 0;
    uint32_t nbytes, nsrc, ndst;
    coll_job_t job{};
    if (rec) {
      if (lane < 2u + COLL_BULK_MAX_SRC + COLL_BULK_MAX_DST) word = __ldg((const unsigned long long *)rec + lane);
      start = __shfl_sync(FULL, word, 0);
      const uint64_t hdr = __shfl_sync(FULL, word, 1);
      nbytes = (uint32_t)hdr;
      nsrc = (uint32_t)(hdr >> 32) & 0xFFFFu;
      ndst = (uint32_t)(hdr >> 48);
    } else {
      const coll_tile_t tile = a.tiles[ti];
      job = a.jobs[tile.job];
      start = tile.start;
      nbytes = tile.nbytes;
      nsrc = job.nsrc;
      ndst = job.ndst;
    }
    if (!waited) griddep_wait();
    waited = true;
    const int64_t ioff = (int64_t)(e % (uint32_t)a.in_pool) * a.in_stride + (int64_t)start;
    const int64_t ooff = (int64_t)e * a.out_stride + (int64_t)start;
    const char *sp = nullptr;
    char *dp = nullptr;
    uint32_t mis = nbytes & 15u;
    if (rec) {
      const uint64_t rs = __shfl_sync(FULL, word, 2u + (lane & 7u));
      const uint64_t rd = __shfl_sync(FULL, word, 2u + COLL_BULK_MAX_SRC + (lane & 7u));
      if (lane < nsrc) {
        sp = a.ptr.in[(uint32_t)(rs >> 56)] + (rs & kOffMask) + ioff;
        mis |= (uint32_t)((uintptr_t)sp & 15u);
      }
      if (lane < ndst) {
        dp = a.ptr.out[(uint32_t)(rd >> 56)] + (rd & kOffMask) + ooff;
        mis |= (uint32_t)((uintptr_t)dp & 15u);
      }
    } else {
      if (lane < nsrc) {
        const coll_ref_t r = a.refs[job.src0 + lane];
        sp = a.ptr.in[r.rank] + r.off + ioff;
        mis |= (uint32_t)((uintptr_t)sp & 15u);
      }
      if (lane < ndst) {
        const coll_ref_t r = a.refs[job.dst0 + lane];
        dp = a.ptr.out[r.rank] + r.off + ooff;
        mis |= (uint32_t)((uintptr_t)dp & 15u);
      }
    }
    const bool slow = __any_sync(FULL, mis != 0) || nsrc > 32 || ndst > 32;
    if (!slow) {
      const uint32_t nvec = nbytes >> 4;
      // The vector loops are warp-uniform (every lane iterates; loads and stores are
      // predicated) because they fetch pointers with full-warp shuffles.
      if constexpr (KIND == 0) {
        const char *s0 = (const char *)__shfl_sync(FULL, (uintptr_t)sp, 0);
        constexpr uint32_t U = 4;
        for (uint32_t base = 0; base < nvec; base += 32 * U) {
          uint4 x[U];
#pragma unroll
          for (uint32_t u = 0; u < U; ++u) {
            const uint32_t idx = base + 32 * u + lane;
            if (idx < nvec) x[u] = zc_load<KIND, KEEP>(s0 + (size_t)idx * 16);
          }
          for (uint32_t d = 0; d < ndst; ++d) {
            char *q = (char *)__shfl_sync(FULL, (uintptr_t)dp, d);
#pragma unroll
            for (uint32_t u = 0; u < U; ++u) {
              const uint32_t idx = base + 32 * u + lane;
              if (idx < nvec) st_cs_v4(q + (size_t)idx * 16, x[u]);
            }
          }
        }
      } else {
        for (uint32_t base = 0; base < nvec; base += 32) {
          const uint32_t v = base + lane;
          const bool act = v < nvec;
          Vec16Acc<KIND - 1> acc;
          for (uint32_t k0 = 0; k0 < nsrc; k0 += 8) {
            uint4 x[8];
            const uint32_t kn = nsrc - k0 < 8 ? nsrc - k0 : 8;
#pragma unroll
            for (uint32_t k = 0; k < 8; ++k) {
              const char *p = (const char *)__shfl_sync(FULL, (uintptr_t)sp, (k0 + k) & 31u);
              if (k < kn && act) x[k] = zc_load<KIND, KEEP>(p + (size_t)v * 16);
            }
            if (act) {
              if constexpr (TREE) {
                tree8<KIND - 1>(acc, k0 == 0, x, kn);
              } else {
#pragma unroll
                for (uint32_t k = 0; k < 8; ++k)
                  if (k < kn) {
                    if (k0 + k == 0) acc.init(x[k]); else acc.add(x[k]);
                  }
              }
            }
          }
          const uint4 r = act ? acc.pack() : make_uint4(0, 0, 0, 0);
          for (uint32_t d = 0; d < ndst; ++d) {
            char *q = (char *)__shfl_sync(FULL, (uintptr_t)dp, d);
            if (act) st_cs_v4(q + (size_t)v * 16, r);
          }
        }
      }
    } else {
      // Element-wise path: pointers recomputed from the tables (or the inline record).
      auto src_of = [&](uint32_t k) {
        if (rec) {
          const uint64_t r = __ldg((const unsigned long long *)rec + 2 + k);
          return (const char *)(a.ptr.in[(uint32_t)(r >> 56)] + (r & kOffMask) + ioff);
        }
        const coll_ref_t r = a.refs[job.src0 + k];
        return (const char *)(a.ptr.in[r.rank] + r.off + ioff);
      };
      auto dst_of = [&](uint32_t d) {
        if (rec) {
          const uint64_t r = __ldg((const unsigned long long *)rec + 2 + COLL_BULK_MAX_SRC + d);
          return a.ptr.out[(uint32_t)(r >> 56)] + (r & kOffMask) + ooff;
        }
        const coll_ref_t r = a.refs[job.dst0 + d];
        return a.ptr.out[r.rank] + r.off + ooff;
      };
      if constexpr (KIND == 0) {
        const char *s0 = src_of(0);
        for (uint32_t i = lane; i < nbytes; i += 32) {
          const char v = s0[i];
          for (uint32_t d = 0; d < ndst; ++d) dst_of(d)[i] = v;
        }
      } else if constexpr (KIND == 1) {
        for (uint32_t i = lane; i < nbytes / 2; i += 32) {
          float acc = __uint_as_float((uint32_t)((const uint16_t *)src_of(0))[i] << 16);
          for (uint32_t k = 1; k < nsrc; ++k)
            acc = __fadd_rn(acc, __uint_as_float((uint32_t)((const uint16_t *)src_of(k))[i] << 16));
          const uint16_t r = (uint16_t)(pack_bf16x2(acc, 0.0f) & 0xFFFFu);
          for (uint32_t d = 0; d < ndst; ++d) ((uint16_t *)dst_of(d))[i] = r;
        }
      } else {
        for (uint32_t i = lane; i < nbytes / 4; i += 32) {
          float acc = ((const float *)src_of(0))[i];
          for (uint32_t k = 1; k < nsrc; ++k) acc = __fadd_rn(acc, ((const float *)src_of(k))[i]);
          for (uint32_t d = 0; d < ndst; ++d) ((float *)dst_of(d))[i] = acc;
        }
      }
    }
  }
}

// ============================================================== staged engine

struct CopyAcc {
  uint4 v;
  __device__ __forceinline__ void init(uint4 x) { v = x; }
  __device__ __forceinline__ void add(uint4) {}
  __device__ __forceinline__ uint4 pack() const { return v; }
};

template <int KIND>
struct EngAcc {
  using type = Vec16Acc<KIND - 1>;
};
template <>
struct EngAcc<0> {
  using type = CopyAcc;
};

__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

__device__ __forceinline__ void spin_ns(uint64_t ns) {
  if (ns == 0) return;
  const uint64_t t0 = globaltimer();
  while (globaltimer() - t0 < ns) {
  }
}

// Poll until `ok(value)`; bounded by the spin limit and by the plan's abort word.
// Returns false on timeout or abort. One lane, one flag.
template <typename Pred>
__device__ __forceinline__ bool spin_u64(const unsigned long long *f, Pred ok,
                                         const coll_dev_status_t *st, uint64_t limit) {
  uint64_t t0 = 0;
  for (uint32_t k = 0;; ++k) {
    const unsigned long long v = ld_acquire_u64(f);
    if (ok(v)) return true;
    if ((k & 31u) == 31u) {
      const uint64_t now = globaltimer();
      if (t0 == 0) t0 = now;
      else if (now - t0 > limit) return false;
      if (ld_relaxed_u32(&st->abort)) return false;
    }
  }
}

__device__ __forceinline__ bool spin_done(const uint32_t *f, uint32_t target,
                                          const coll_dev_status_t *st, uint64_t limit) {
  uint64_t t0 = 0;
  for (uint32_t k = 0;; ++k) {
    const uint32_t v = ld_acquire_u32(f);
    if ((int32_t)(v - target) >= 0) return true;
    if ((k & 31u) == 31u) {
      const uint64_t now = globaltimer();
      if (t0 == 0) t0 = now;
      else if (now - t0 > limit) return false;
      if (ld_relaxed_u32(&st->abort)) return false;
    }
  }
}

__device__ void record_timeout(coll_dev_status_t *st, int rank, int unit, int where,
                               uint32_t epoch) {
  if (atomicCAS(&st->status, 0, COLL_ETIMEDOUT) == 0) {
    st->fail_rank = rank;
    st->fail_unit = unit;
    st->fail_where = where;
    st->fail_epoch = epoch;
  }
  st_relaxed_u32(&st->abort, 1u);
}

// A producer slot's flag word: {epoch mod 2^16 : 16 | tag B mod 2^16 : 16 | tag A : 32},
// written with one 64-bit store. Flags of one slot only ever hold E or an epoch one or two
// before it, so 16 bits of epoch tell them apart across any wrap.
__device__ __forceinline__ unsigned long long flag_word(uint32_t E, uint32_t ta, uint32_t tb) {
  return ((unsigned long long)(E & 0xFFFFu) << 48) | ((unsigned long long)(tb & 0xFFFFu) << 32) |
         ta;
}
__device__ __forceinline__ uint32_t flag_epoch(unsigned long long f) { return (uint32_t)(f >> 48); }
__device__ __forceinline__ bool flag_is(unsigned long long f, uint32_t E) {
  return flag_epoch(f) == (E & 0xFFFFu);
}

// Wait (all lanes cooperating) until every producer flag of a unit carries epoch E.
__device__ __forceinline__ bool wait_producers(const unsigned long long *pf, uint32_t n,
                                               uint32_t E, const coll_dev_status_t *st,
                                               uint64_t limit) {
  const uint32_t lane = threadIdx.x & 31u;
  bool ok = true;
  for (uint32_t j = lane; j < n; j += 32)
    ok = ok && spin_u64(pf + j, [E](unsigned long long v) { return flag_is(v, E); },
                        st, limit);
  return __all_sync(FULL, ok);
}

__device__ __forceinline__ bool wait_consumers_done(const uint32_t *cf, uint32_t n,
                                                    uint32_t target,
                                                    const coll_dev_status_t *st,
                                                    uint64_t limit) {
  const uint32_t lane = threadIdx.x & 31u;
  bool ok = true;
  for (uint32_t j = lane; j < n; j += 32) ok = ok && spin_done(cf + j, target, st, limit);
  return __all_sync(FULL, ok);
}

// Reduce (or copy) the n pieces of a unit in slot order, loads in batches of 8 so that
// every batch's loads are in flight together.
template <int KIND>
__device__ __forceinline__ uint4 gather_pieces(const char *xb, uint32_t nbytes, uint32_t n,
                                               uint32_t lane, bool active) {
  typename EngAcc<KIND>::type acc;
  for (uint32_t k0 = 0; k0 < n; k0 += 8) {
    uint4 x[8];
    const uint32_t kn = n - k0 < 8 ? n - k0 : 8;
#pragma unroll
    for (uint32_t k = 0; k < 8; ++k)
      if (k < kn && active) x[k] = ld_relaxed_v4(xb + (size_t)(k0 + k) * nbytes + lane * 16);
    if (active) {
#pragma unroll
      for (uint32_t k = 0; k < 8; ++k)
        if (k < kn) {
          if (k0 + k == 0) acc.init(x[k]); else acc.add(x[k]);
        }
    }
  }
  return active ? acc.pack() : make_uint4(0, 0, 0, 0);
}

// ------------------------------------------------------------------ fused producer
// The fused-producer variant computes each rank's payload piece as y = W_r x in the stage
// step: for every output column, the k products (rounded to binary32) added in row order
// from the first one, then rounded once to bf16 — the plain definition of the dot product,
// in the order it is written. A CTA runs eight warps:
//   warp 0      the engine warp (the staged protocol, unchanged);
//   warp 1      the weight streamer: lane 0 fills a ring of shared-memory slots, each one
//               tensor copy (TMA) of 64 rows x the unit's columns (at most 256) of W_r, for
//               the pieces of the whole run in order (the weights do not depend on the
//               epoch's data, so it runs ahead by as many slots as the ring holds, across
//               exchanges);
//   warp 2      the x streamer: lane 0 copies piece q's x (k bf16, one bulk copy) into one
//               of two buffers, once the engine has opened piece q (that also frees the
//               buffer: piece q is opened only after piece q - 2 was taken, whose x was read
//               before its results were written);
//   warp 3      idle;
//   warps 4..7  compute warps: lane l of compute warp w owns columns 64w + 2l and
//               64w + 2l + 1 of the piece (lanes past the unit's columns idle) and carries
//               their two chains over all k rows (packed binary32 pairs), so no order is
//               split; it writes the rounded results into one of two result slots.
// The engine takes piece q's results from its slot and opens piece q + 2 (at most one
// piece computed ahead; the result slot of piece q + 2 is the one just taken): without chained epochs the next piece is computed while the
// engine runs the current exchange. With chained epochs an epoch's pieces are opened only
// after the rank's previous epoch is complete, as the next layer's input would depend on it.
// Every wait is bounded by the plan's spin limit and stops on the abort word or when the
// engine ends the run; the streamers then wait (bounded) for the copies they issued.
constexpr uint32_t kGemvComputeWarps = 4;
constexpr uint32_t kGemvFirst = 4;                        // warp of compute warp 0
constexpr uint32_t kGemvThreads = 32 * (kGemvFirst + kGemvComputeWarps);  // 256
constexpr uint32_t kGemvRows = 64;                        // weight rows per slot (one copy)
constexpr uint32_t kGemvMaxPitch = 512;                   // bytes per staged row, at most
constexpr uint32_t kGemvRingBytes = 168u << 10;           // the ring: 5 slots of 512-byte
                                                          // rows, 6 of 432, at most 8
constexpr uint32_t kGemvMaxSlots = 8;
constexpr uint32_t kGemvMaxK = 8192;                      // rows of W_r (length of x)
constexpr uint32_t kGemvXBytes = 2 * kGemvMaxK;
constexpr uint32_t kGemvMaxItems = 16;                    // stage items whose rows are cached
// dynamic shared memory: ring, two x buffers, two result slots, barriers (+128 for the
// alignment of the ring, where the tensor copies land)
constexpr uint32_t kGemvBars = 2 * kGemvMaxSlots + 4;
constexpr uint32_t kGemvSmemBytes =
    kGemvRingBytes + 2 * kGemvXBytes + 2 * kGemvMaxPitch + kGemvBars * 8 + 128;

struct GemvShared {
  uint64_t go;          // pieces the compute may start (written by warp 0, release.cta)
  uint64_t chain_open;  // with chained epochs: pieces of the epochs already allowed
  uint64_t total;       // pieces of the run (epochs x items)
  uint64_t taken;       // pieces whose results warp 0 has taken
  uint32_t exit;        // set by warp 0 when its loop ends: the other roles stop
  uint32_t nitems;      // stage items of this warp, in order
  uint32_t kslots;      // slots per piece (k / 64, rounded up)
  uint32_t k;
  const CUtensorMap *maps;                 // W_r of each rank (kernel parameters)
  const CUtensorMap *wmap[kGemvMaxItems];  // each cached item's matrix ...
  uint32_t wcol[kGemvMaxItems];            // ... its first column ...
  uint32_t wrank[kGemvMaxItems];           // ... and its rank (the x buffer's owner)
};

__device__ __forceinline__ GemvShared &gemv_smem() {
  __shared__ GemvShared g;
  return g;
}

struct GemvBufs {
  unsigned char *ring;  // [gemv_slots][kGemvRows][gemv_pitch]
  unsigned char *x;     // [2][kGemvXBytes]
  unsigned char *res;   // [2][kGemvMaxPitch]
  uint64_t *full;       // [kGemvMaxSlots] a fill's rows have landed
  uint64_t *empty;      // [kGemvMaxSlots] every compute warp has read the slot
  uint64_t *xfull;      // [2] piece's x has landed
  uint64_t *rfull;      // [2] every compute warp has written its results
};

__device__ __forceinline__ GemvBufs gemv_bufs() {
  extern __shared__ __align__(128) unsigned char gemv_dyn[];
  GemvBufs b;
  b.ring = gemv_dyn + ((128u - (smem_u32(gemv_dyn) & 127u)) & 127u);
  b.x = b.ring + kGemvRingBytes;
  b.res = b.x + 2 * kGemvXBytes;
  b.full = reinterpret_cast<uint64_t *>(b.res + 2 * kGemvMaxPitch);
  b.empty = b.full + kGemvMaxSlots;
  b.xfull = b.empty + kGemvMaxSlots;
  b.rfull = b.xfull + 2;
  return b;
}

__device__ __forceinline__ uint64_t ld_acquire_cta_shared(const uint64_t *p) {
  uint64_t v;
  asm volatile("ld.acquire.cta.shared.u64 %0, [%1];" : "=l"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_cta_shared(uint64_t *p, uint64_t v) {
  asm volatile("st.release.cta.shared.u64 [%0], %1;" ::"r"(smem_u32(p)), "l"(v) : "memory");
}
__device__ __forceinline__ void st_release_cta_shared(uint32_t *p, uint32_t v) {
  asm volatile("st.release.cta.shared.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

// The bound on the waits of the streamers and the compute warps. They wait on the engine warp
// of their CTA (directly or through each other), whose own waits are bounded by the spin
// limit and which ends the run (or records the timeout) when one expires; a longer bound
// here keeps a slow but live engine from being reported as a timeout of another role.
__device__ __forceinline__ uint64_t gemv_role_limit(const EngArgs &a) {
  return a.spin_ns > (~0ull >> 4) ? ~0ull : a.spin_ns << 4;
}

// Stop polling: the engine ended the run, or some warp of the plan gave up.
__device__ __forceinline__ bool gemv_stop(const EngArgs &a) {
  const GemvShared &g = gemv_smem();
  return *reinterpret_cast<const volatile uint32_t *>(&g.exit) != 0u ||
         ld_relaxed_u32(&a.st->abort) != 0u;
}

// Where piece q's rows and x come from (cached for the first items).
struct GemvSrc {
  const CUtensorMap *map;
  uint32_t col;
  uint32_t rank;
};

__device__ __forceinline__ GemvSrc gemv_item(const EngArgs &a, const GemvShared &g,
                                             const coll_warp_t &W, uint32_t idx) {
  if (idx < kGemvMaxItems) return GemvSrc{g.wmap[idx], g.wcol[idx], g.wrank[idx]};
  const coll_item_t it = a.sitems[W.s0 + idx];
  const coll_unit_t u = a.units[it.unit];
  const coll_ref_t r = a.refs[u.src0 + it.slot];
  return GemvSrc{g.maps + r.rank, (uint32_t)((r.off + u.start) >> 1), r.rank};
}

// Warp 0, before the role split: cache the stage items' row sources and the run's sizes,
// and open the first pieces.
__device__ void gemv_prologue(const EngArgs &a, const CUtensorMap *maps, const coll_warp_t &W,
                              bool chained, uint32_t lane) {
  GemvShared &g = gemv_smem();
  const uint32_t nitems = W.s1 - W.s0;
  if (lane == 0) {
    g.nitems = nitems;
    g.k = a.gemv_k;
    g.kslots = (a.gemv_k + kGemvRows - 1u) / kGemvRows;
    g.total = (uint64_t)a.n_epochs * nitems;
    g.maps = maps;
    g.exit = 0;
    g.taken = 0;
    g.chain_open = chained ? 0u : ~0ull;
    g.go = chained ? 0u : (g.total < 2u ? g.total : 2u);
  }
  for (uint32_t idx = lane; idx < nitems && idx < kGemvMaxItems; idx += 32) {
    const coll_item_t it = a.sitems[W.s0 + idx];
    const coll_unit_t u = a.units[it.unit];
    const coll_ref_t r = a.refs[u.src0 + it.slot];
    g.wmap[idx] = maps + r.rank;
    g.wcol[idx] = (uint32_t)((r.off + u.start) >> 1);
    g.wrank[idx] = r.rank;
  }
}

// Warp 0: open pieces up to min(taken + 2, chain_open) for the x streamer and the compute.
__device__ __forceinline__ void gemv_open(GemvShared &g) {
  const uint64_t lim = g.taken + 2ull < g.chain_open ? g.taken + 2ull : g.chain_open;
  st_release_cta_shared(&g.go, lim < g.total ? lim : g.total);
}

// Warp 1, lane 0: every weight fill of the run in order; fill f lands in slot f % S once
// the compute warps have released that slot's previous fill. A last fill past row k reads
// zeros (the rows lie outside the tensor map) and is only partly used.
__device__ void gemv_weight_streamer(const EngArgs &a, const coll_warp_t &W) {
  GemvShared &g = gemv_smem();
  const GemvBufs b = gemv_bufs();
  const uint64_t fills = g.total * g.kslots;
  const uint32_t S = a.gemv_slots, slot_bytes = kGemvRows * a.gemv_pitch;
  uint64_t f = 0;
  uint32_t s = 0, lap = 0, j = 0, item = 0;
  GemvSrc src = gemv_item(a, g, W, 0);
  bool ok = true;
  for (; f < fills; ++f) {
    ok = mbar_wait_until(&b.empty[s], (lap & 1u) ^ 1u, gemv_role_limit(a),
                         [&a]() { return gemv_stop(a); });
    if (!ok) break;
    mbar_expect_tx(&b.full[s], slot_bytes);
    tensor_load_2d(b.ring + (size_t)s * slot_bytes, src.map, src.col, j * kGemvRows, &b.full[s]);
    if (++s == S) {
      s = 0;
      ++lap;
    }
    if (++j == g.kslots) {
      j = 0;
      if (++item == g.nitems) item = 0;
      src = gemv_item(a, g, W, item);
    }
  }
  if (!ok && !gemv_stop(a)) record_timeout(a.st, (int)W.rank, -1, 6, 0);
  // every fill issued has landed before the CTA may exit (bounded): the last fill of each
  // slot is the latest phase of its barrier
  const uint64_t issued = f;
  for (uint32_t t = 0; t < S && (uint64_t)t < issued; ++t) {
    const uint64_t last = issued - 1u - ((issued - 1u - t) % S);
    mbar_wait_until(&b.full[t], (uint32_t)((last / S) & 1u), 100000000ull,
                    []() { return false; });
  }
}

// Warp 2, lane 0: piece q's x (k bf16) into buffer q % 2, once the engine has opened piece
// q (so the buffer's previous piece, q - 2, has been read and its results taken). The
// acquire here and the release of the copy's arrival order the compute lanes' reads of the
// result slot after the engine's, through the x barrier they wait on.
__device__ void gemv_x_streamer(const EngArgs &a, const coll_warp_t &W) {
  GemvShared &g = gemv_smem();
  const GemvBufs b = gemv_bufs();
  const uint32_t xbytes = g.k * 2u;
  uint64_t q = 0;
  uint32_t item = 0, pool = 0;
  bool ok = true;
  for (; q < g.total; ++q) {
    // wait until the engine opens piece q
    uint64_t t0 = 0;
    for (uint32_t it = 0; ld_acquire_cta_shared(&g.go) <= q; ++it) {
      __nanosleep(64);  // (polling at full rate would take issue slots from a compute warp)
      if ((it & 15u) == 15u) {
        const uint64_t now = globaltimer();
        if (t0 == 0) t0 = now;
        else if (now - t0 > gemv_role_limit(a)) ok = false;
        if (!ok || gemv_stop(a)) break;
      }
    }
    if (!ok || ld_acquire_cta_shared(&g.go) <= q) break;
    const uint32_t p = (uint32_t)(q & 1u);
    const GemvSrc src = gemv_item(a, g, W, item);
    const char *xp = a.ptr.in[src.rank] + (int64_t)pool * a.in_stride;
    mbar_expect_tx(&b.xfull[p], xbytes);
    bulk_load(b.x + (size_t)p * kGemvXBytes, xp, xbytes, &b.xfull[p]);
    if (++item == g.nitems) {
      item = 0;
      if (++pool == (uint32_t)a.in_pool) pool = 0;
    }
  }
  if (!ok && !gemv_stop(a)) record_timeout(a.st, (int)W.rank, -1, 6, 0);
  for (uint64_t t = q > 2 ? q - 2 : 0; t < q; ++t)
    mbar_wait_until(&b.xfull[t & 1u], (uint32_t)((t >> 1) & 1u), 100000000ull,
                    []() { return false; });
}

// Packed pairs of binary32 (sm_100 family): two IEEE operations, round to nearest even.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// The products of sixteen rows for this lane's two columns: prod[r] = w[row][c..c+1] * x[row]
// (each rounded to binary32), independent of the running sums. PITCH: bytes per staged row
// when known at compile time (the rows' offsets are then immediates of the loads), else 0
// and `pitch` gives it.
template <uint32_t PITCH>
__device__ __forceinline__ void gemv_prods16(uint64_t prod[16], const unsigned char *slot,
                                             uint32_t pitch, uint32_t colb,
                                             const unsigned char *xrow) {
  if constexpr (PITCH != 0) pitch = PITCH;
  const uint4 xa = *reinterpret_cast<const uint4 *>(xrow);
  const uint4 xb = *reinterpret_cast<const uint4 *>(xrow + 16);
  const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
  for (uint32_t r = 0; r < 16; ++r) {
    const uint32_t w = *reinterpret_cast<const uint32_t *>(slot + r * pitch + colb);
    const float xf = __uint_as_float((r & 1u) ? (xw[r >> 1] & 0xFFFF0000u) : (xw[r >> 1] << 16));
    prod[r] = f2_mul(f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u)),
                     f2_pack(xf, xf));
  }
}

// The running sums over sixteen products in row order (FIRST: the chain starts from the
// first of them).
template <bool FIRST>
__device__ __forceinline__ void gemv_adds16(uint64_t &acc, const uint64_t prod[16]) {
#pragma unroll
  for (uint32_t r = 0; r < 16; ++r) acc = (FIRST && r == 0) ? prod[r] : f2_add(acc, prod[r]);
}

// BLOCKS blocks of sixteen rows of a slot, in order: the products of block c + 1 are formed
// while block c's sums run (they do not depend on them), so the in-order chain of adds has
// independent work to overlap; the order of the adds is unchanged.
template <bool FIRST, uint32_t BLOCKS, uint32_t PITCH>
__device__ __forceinline__ void gemv_slot_rows(uint64_t &acc, const unsigned char *slot,
                                               uint32_t pitch, uint32_t colb,
                                               const unsigned char *xs) {
  if constexpr (PITCH != 0) pitch = PITCH;
  uint64_t prod[2][16];
  gemv_prods16<PITCH>(prod[0], slot, pitch, colb, xs);
#pragma unroll
  for (uint32_t c = 0; c < BLOCKS; ++c) {
    if (c + 1 < BLOCKS)
      gemv_prods16<PITCH>(prod[(c + 1) & 1], slot + (c + 1) * 16 * pitch, pitch, colb,
                          xs + (c + 1) * 32);
    if (FIRST && c == 0) gemv_adds16<true>(acc, prod[c & 1]);
    else gemv_adds16<false>(acc, prod[c & 1]);
  }
}

// The rows of one fill: 64, or fewer (a multiple of 16) in a last fill past row k.
template <bool FIRST, uint32_t PITCH>
__device__ __forceinline__ void gemv_fill_rows(uint64_t &acc, const unsigned char *slot,
                                               uint32_t pitch, uint32_t colb,
                                               const unsigned char *xs, uint32_t rows) {
  switch (rows) {
    case 16: gemv_slot_rows<FIRST, 1, PITCH>(acc, slot, pitch, colb, xs); break;
    case 32: gemv_slot_rows<FIRST, 2, PITCH>(acc, slot, pitch, colb, xs); break;
    case 48: gemv_slot_rows<FIRST, 3, PITCH>(acc, slot, pitch, colb, xs); break;
    default: gemv_slot_rows<FIRST, 4, PITCH>(acc, slot, pitch, colb, xs); break;
  }
}

// Compute warp `cw` (0..3): every piece of the run in order. Waits are taken by lane 0 and
// shared; a __syncwarp after each orders lane 0's acquiring wait before every lane's reads,
// and one before each of lane 0's arrivals orders every lane's reads (of a slot) or writes
// (of results) before it.
template <uint32_t PITCH>
__device__ void gemv_compute(const EngArgs &a, const coll_warp_t &W, uint32_t cw,
                             uint32_t lane) {
  GemvShared &g = gemv_smem();
  const GemvBufs b = gemv_bufs();
  const uint32_t colb = (64u * cw + 2u * lane) * 2u;  // byte offset of this lane's columns
  const uint32_t pitch = PITCH ? PITCH : a.gemv_pitch, S = a.gemv_slots;
  const uint32_t slot_bytes = kGemvRows * pitch;
  const bool live = PITCH == kGemvMaxPitch || colb < pitch;  // columns inside the unit
  uint32_t s = 0, lap = 0;
  bool ok = true;
  for (uint64_t q = 0; q < g.total && ok; ++q) {
    const uint32_t p = (uint32_t)(q & 1u);
    if (lane == 0)
      ok = mbar_wait_until(&b.xfull[p], (uint32_t)((q >> 1) & 1u), gemv_role_limit(a),
                           [&a]() { return gemv_stop(a); });
    ok = __shfl_sync(FULL, ok, 0);
    __syncwarp();
    if (!ok) break;
    const unsigned char *xq = b.x + (size_t)p * kGemvXBytes;
    uint64_t acc = 0;
    for (uint32_t j = 0; j < g.kslots; ++j) {
      if (lane == 0)
        ok = mbar_wait_until(&b.full[s], lap & 1u, gemv_role_limit(a),
                             [&a]() { return gemv_stop(a); });
      ok = __shfl_sync(FULL, ok, 0);
      __syncwarp();
      if (!ok) break;
      const unsigned char *slot = b.ring + (size_t)s * slot_bytes;
      const unsigned char *xs = xq + (size_t)j * (kGemvRows * 2);
      // rows of this fill: 64, or fewer (a multiple of 16) in a last fill past row k
      const uint32_t rows = g.k - j * kGemvRows < kGemvRows ? g.k - j * kGemvRows : kGemvRows;
      if (live) {
        if (j == 0) gemv_fill_rows<true, PITCH>(acc, slot, pitch, colb, xs, rows);
        else gemv_fill_rows<false, PITCH>(acc, slot, pitch, colb, xs, rows);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&b.empty[s]);  // the warp's reads of the slot are done
      if (++s == S) {
        s = 0;
        ++lap;
      }
    }
    if (!ok) break;
    // piece q's x has landed, so the engine has opened piece q: it has taken piece q - 2
    // from this result slot (its release of the opening, the streamer's acquire and the
    // x barrier order that before these writes)
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(acc));
    if (live)
      *reinterpret_cast<uint32_t *>(b.res + (size_t)p * kGemvMaxPitch + colb) = pack_bf16x2(lo, hi);
    __syncwarp();
    if (lane == 0) mbar_arrive(&b.rfull[p]);
  }
  if (!ok && lane == 0 && !gemv_stop(a)) record_timeout(a.st, (int)W.rank, -1, 6, 0);
}

// Warp 0 (all 32 lanes): take piece q's results (lanes below `active` hold 8 outputs each)
// and open piece q + 2; false if the wait gave up.
__device__ __forceinline__ bool gemv_take(const EngArgs &a, uint64_t q, uint32_t active,
                                          uint32_t lane, uint4 &res) {
  GemvShared &g = gemv_smem();
  const GemvBufs b = gemv_bufs();
  const uint32_t p = (uint32_t)(q & 1u);
  bool ok = true;
  if (lane == 0)
    ok = mbar_wait_until(&b.rfull[p], (uint32_t)((q >> 1) & 1u), a.spin_ns,
                         [&a]() { return ld_relaxed_u32(&a.st->abort) != 0u; });
  ok = __shfl_sync(FULL, ok, 0);
  __syncwarp();
  if (!ok) return false;
  res = lane < active ? *reinterpret_cast<const uint4 *>(b.res + (size_t)p * kGemvMaxPitch + lane * 16)
                      : make_uint4(0, 0, 0, 0);
  __syncwarp();  // every lane's read of the slot precedes lane 0's release of it
  if (lane == 0) {
    g.taken = q + 1u;
    gemv_open(g);
  }
  return true;
}

// Warp 0, at an epoch whose chained wait has passed: open that epoch's pieces.
__device__ __forceinline__ void gemv_open_epoch(uint32_t epoch_index, uint32_t lane) {
  GemvShared &g = gemv_smem();
  if (lane == 0) {
    g.chain_open = (uint64_t)(epoch_index + 1u) * g.nitems;
    gemv_open(g);
  }
}

// Warp 0 at the end of its loop: the other roles stop waiting.
__device__ __forceinline__ void gemv_finish(uint32_t lane) {
  GemvShared &g = gemv_smem();
  if (lane == 0) st_release_cta_shared(&g.exit, 1u);
}

// Validation of a speculative load: lane j < n holds producer j's flag word and every lane
// holds its share of the two hashes of what it loaded. Passes iff every flag shows epoch E
// and, for each tag, the producers' tags (hash + E*K each) add up to the loaded hash plus
// n*E*K (tag A modulo 2^32, tag B modulo 2^16), i.e. the loaded bytes are the notified
// bytes up to a 48-bit collision.
__device__ __forceinline__ bool tags_match(unsigned long long f, uint2 myh, uint32_t n,
                                           uint32_t E, uint32_t lane) {
  const uint32_t fta = __reduce_add_sync(FULL, lane < n ? (uint32_t)f : 0u);
  const uint32_t ftb = __reduce_add_sync(FULL, lane < n ? (uint32_t)(f >> 32) & 0xFFFFu : 0u);
  const uint2 h = reduce_add2(myh);
  const bool epochs = __all_sync(FULL, lane >= n || flag_is(f, E));
  return epochs && fta == h.x + n * tag_fold(0u, E) &&
         ((ftb - (h.y + n * tag_fold_b(0u, E))) & 0xFFFFu) == 0u;
}

// If `side` is set, the warp also hashes `side_v` (the prefetched next input piece, lanes
// below side_nvec) into side_h while the first batch of loads is in flight.
template <int KIND>
__device__ __forceinline__ uint4 spec_attempt(const char *xb, uint32_t nbytes, uint32_t n,
                                              uint32_t lane, bool active, bool want_hash,
                                              const unsigned long long *pf, bool acquire_flags,
                                              bool load_flags, unsigned long long &f,
                                              uint2 &myh, bool side, uint4 side_v,
                                              uint32_t side_nvec, uint2 &side_h) {
  typename EngAcc<KIND>::type acc;
  myh = make_uint2(0u, 0u);
  for (uint32_t k0 = 0; k0 < n; k0 += 8) {
    uint4 x[8];
    const uint32_t kn = n - k0 < 8 ? n - k0 : 8;
#pragma unroll
    for (uint32_t k = 0; k < 8; ++k)
      x[k] = (k < kn && active) ? ld_relaxed_v4(xb + (size_t)(k0 + k) * nbytes + lane * 16)
                                : make_uint4(0, 0, 0, 0);
    if (k0 == 0 && load_flags && lane < n)
      f = acquire_flags ? ld_acquire_u64(pf + lane) : ld_relaxed_u64(pf + lane);
    if (k0 == 0 && side)
      side_h = reduce_add2(lane < side_nvec ? tag_part(side_v, lane) : make_uint2(0u, 0u));
    if (active) {
#pragma unroll
      for (uint32_t k = 0; k < 8; ++k)
        if (k < kn) {
          if (k0 + k == 0) acc.init(x[k]); else acc.add(x[k]);
        }
    }
    if (want_hash && active) {
      // this lane's share of every producer's hashes, summed: the check compares totals
      const uint2 h = tag_parts8(x, kn, lane);
      myh.x += h.x;
      myh.y += h.y;
    }
  }
  return active ? acc.pack() : make_uint4(0, 0, 0, 0);
}

// KIND: 0 copy, 1 sum of bf16, 2 sum of f32. GEMV: fused producer. LL: tagged data.
// PULL: two-shot pull plans (the publish/pull steps are compiled only into this variant).
// FP: 0 for the general engine; otherwise a variant for plans whose every warp has one
// stage item and one consume item, run without fault injection or phase stamps, under one
// speculative protocol known at compile time (1 with content tags, 2 the same fence-free;
// 3 and 4 the same two with one %globaltimer stamp per epoch, so that the latency
// distribution is taken on the specialised code; 5 and 6 the same two with chained epochs). On the single warp that carries a
// piece through an epoch, every runtime mode test is a dependent instruction on the critical
// path; compiled out, the decode epoch drops by about a sixth. (A dual-buffer variant
// measured slower than the general engine and is not built.)
// (the fused producer also takes the tensor maps of the ranks' weight matrices)
template <bool GEMV> struct MapsArg { using type = NoMaps; };
template <> struct MapsArg<true> { using type = GemvMaps; };

template <int KIND, bool GEMV, bool LL, bool PULL, int FP>
__global__ void __launch_bounds__(GEMV ? kGemvThreads : 32, 1)
    engine_kernel(const EngArgs a, const __grid_constant__ typename MapsArg<GEMV>::type maps) {
  static_assert(FP == 0 || (!GEMV && !LL && !PULL), "the specialised variants are plain");
  constexpr bool fast = FP != 0;
  constexpr bool fp_relaxed = FP == 2 || FP == 4 || FP == 6;  // the fence-free check
  constexpr bool fp_stamps = FP == 3 || FP == 4;  // ... with one stamp per epoch
  constexpr bool fp_chain = FP >= 5;              // ... with chained epochs
  const uint32_t gw = blockIdx.x;
  const uint32_t lane = threadIdx.x & 31u;
  if constexpr (GEMV) {
    const uint32_t wid = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
      const GemvBufs bb = gemv_bufs();
      for (uint32_t s = 0; s < kGemvMaxSlots; ++s) {
        mbar_init(&bb.full[s], 1);  // the streamer's arrival, plus the copy's bytes
        mbar_init(&bb.empty[s], kGemvComputeWarps);
      }
      for (uint32_t p = 0; p < 2; ++p) {
        mbar_init(&bb.xfull[p], 1);
        mbar_init(&bb.rfull[p], kGemvComputeWarps);
      }
      mbar_init_fence();
    }
    __syncthreads();
    if (gw >= a.nwarps) return;  // (every CTA of a launch is a plan warp)
    if (wid == 0) gemv_prologue(a, maps.m, a.warps[gw], a.chain && a.rank_done, lane);
    __syncthreads();  // the item cache, the run's sizes and the first opened pieces are set
    if (wid == 1) {
      if (lane == 0) gemv_weight_streamer(a, a.warps[gw]);
      return;
    }
    if (wid == 2) {
      if (lane == 0) gemv_x_streamer(a, a.warps[gw]);
      return;
    }
    if (wid >= kGemvFirst) {
      // the two unit sizes in use get the rows' offsets compiled in
      if (a.gemv_pitch == 512) gemv_compute<512>(a, a.warps[gw], wid - kGemvFirst, lane);
      else if (a.gemv_pitch == 432) gemv_compute<432>(a, a.warps[gw], wid - kGemvFirst, lane);
      else gemv_compute<0>(a, a.warps[gw], wid - kGemvFirst, lane);
      return;
    }
    if (wid != 0) return;
  } else {
    if (gw >= a.nwarps) return;
  }
  const coll_warp_t W = a.warps[gw];
  coll_dev_status_t *st = a.st;
  const bool spec_proto = fast || a.protocol == COLL_PROTO_SPEC;
  const bool barrier_proto = !fast && a.protocol == COLL_PROTO_BARRIER;
  constexpr bool ll = LL;
  const uint32_t slot_mult = ll ? 2u : 1u;  // tagged-data slots are twice the payload
  // content tags: validated by the tagged checks, stored by every spec producer
  const bool literal = !fast && spec_proto && a.spec_check == COLL_SPEC_LITERAL;
  const bool relaxed = fast ? fp_relaxed : spec_proto && a.spec_check == COLL_SPEC_TAGGED_RELAXED;
  const bool tagged = spec_proto && !literal;
  const bool skip_notify = !fast && (a.inject_flags & COLL_INJECT_SKIP_NOTIFY) &&
                           (int)W.rank == a.inject_rank;
  const bool pause_consumer = !fast && (a.inject_flags & COLL_INJECT_SPEC_PAUSE) &&
                              (int)W.rank == a.inject_rank;
  const bool delay_producer = !fast && (a.inject_flags & COLL_INJECT_SPEC_PAUSE) &&
                              (int)W.rank == (a.inject_rank + 1) % a.R;
  const bool chained = fast ? fp_chain : a.chain && a.rank_done;
  const bool stagger = !fast && (a.inject_flags & COLL_INJECT_STAGGER);
  uint32_t n_checks = 0, n_retries = 0;
  uint32_t win = a.spec_delay_ns << 3;  // the speculation window of this warp (ns / 8)
  bool failed = false;
  uint64_t gpiece = 0;  // fused producer: pieces computed so far

  // A warp with exactly one stage item prefetches the next epoch's input piece (read-only
  // during the kernel) and hashes it while its own consume waits on memory, which takes
  // the input load and the producer-side tag off the critical path.
  constexpr bool gemv = GEMV;
  const bool single_s = fast || (W.s1 - W.s0) == 1u;
  const uint32_t s_end = fast ? W.s0 + 1u : W.s1;
  const bool pipelined = single_s && !gemv;
  coll_unit_t su;
  coll_ref_t sref;
  coll_item_t sit;
  // A warp with a single consume item (the all-reduce case) also keeps that item, its
  // unit and its output reference in registers: the plan tables are then read once, not
  // once per epoch (acquire loads may invalidate L1, which would make every table read an
  // L2 round trip on the critical path).
  const bool single_c = fast || (W.c1 - W.c0) == 1u;
  const uint32_t c_end = fast ? W.c0 + 1u : W.c1;
  coll_item_t cit;
  coll_unit_t cu;
  coll_ref_t cref;
  if (single_c) {
    cit = a.citems[W.c0];
    cu = a.units[cit.unit];
    cref = a.refs[cu.dst0 + (cit.slot == COLL_SLOT_ALL ? 0u : cit.slot)];
  }
  uint4 nx = make_uint4(0, 0, 0, 0);
  uint2 nh = make_uint2(0u, 0u);
  bool nh_ready = false;
  const char *sin_base = nullptr;  // single stage item: its input piece at pool entry 0
  char *cout_base = nullptr;        // single consume item: its output piece at epoch 0
  if (single_c) cout_base = a.ptr.out[cref.rank] + cref.off + cu.start;
  if (single_s) {
    sit = a.sitems[W.s0];
    su = a.units[sit.unit];
    sref = a.refs[su.src0 + sit.slot];
  }
  if (pipelined) {
    sin_base = a.ptr.in[sref.rank] + sref.off + su.start;
    if (lane < (su.nbytes >> 4) && a.n_epochs > 0)
      nx = ld_nc_v4(a.ptr.in[sref.rank] + sref.off + su.start + lane * 16);
  }

  if (stagger && a.inject_start_ns)
    spin_ns((uint64_t)W.rank * a.inject_start_ns);
  const bool stamp = (!fast || fp_stamps) && gw == 0 && lane == 0 && a.stamps;
  const bool phases = !fast && stamp && a.stamp_phases;
  if (stamp) a.stamps[0] = globaltimer();

  // input-pool offset of epoch i and of epoch i+1, advanced without division (a runtime
  // modulo costs a long dependent chain on this single-warp critical path)
  int64_t in_off = 0, in_off_next = a.in_pool > 1 ? a.in_stride : 0;
  int32_t pool_next = a.in_pool > 1 ? 1 : 0;
  for (int i = 0; i < a.n_epochs && !failed; ++i) {
    const uint32_t E = a.epoch_base + (uint32_t)i + 1u;
    const uint32_t b = barrier_proto ? 0u : (E & 1u);
    if (i > 0) {
      in_off = in_off_next;
      pool_next = pool_next + 1 == a.in_pool ? 0 : pool_next + 1;
      in_off_next = (int64_t)pool_next * a.in_stride;
    }
    const int64_t out_off = (int64_t)i * a.out_stride;

    if (stagger && a.inject_prob_ppm) {
      const uint64_t h = splitmix64(a.inject_seed ^ ((uint64_t)E * 0xD1B54A32D192ED03ull));
      if ((h % 1000000ull) < a.inject_prob_ppm && W.rank == (uint32_t)((h >> 40) % (uint64_t)a.R))
        spin_ns(splitmix64(h) % (a.inject_max_ns + 1));
    }

    const bool pst = phases && (uint32_t)i < a.stamp_cap;
    if (chained) {
      // dependent chain: wait until every warp of this rank finished epoch E-1's consume
      bool ok = true;
      if (lane == 0) {
        const uint32_t target = W.rank_warps * (E - 1u);
        uint64_t t0 = 0;
        for (uint32_t k = 0; (int32_t)(ld_acquire_u32(a.rank_done + W.rank) - target) < 0; ++k) {
          if ((k & 31u) == 31u) {
            const uint64_t now = globaltimer();
            if (t0 == 0) t0 = now;
            else if (now - t0 > a.spin_ns || ld_relaxed_u32(&st->abort)) {
              ok = false;
              break;
            }
          }
        }
      }
      if (!__all_sync(FULL, __shfl_sync(FULL, ok, 0))) {
        if (lane == 0) record_timeout(st, (int)W.rank, -1, 4, E);
        failed = true;
        break;
      }
      if constexpr (GEMV) gemv_open_epoch((uint32_t)i, lane);  // this epoch's inputs are ready
    }
    if (pst) a.stamps[1 + 4 * i] = globaltimer();

    // ---------------- Stage + Notify
    for (uint32_t s = W.s0; s < s_end; ++s) {
      const coll_item_t it = single_s ? sit : a.sitems[s];
      const coll_unit_t u = single_s ? su : a.units[it.unit];
      if (barrier_proto || (u.flags & COLL_UNIT_REUSE_WAIT)) {
        // bottom barrier (single buffer) / explicit reuse wait (dual buffers)
        const uint32_t target = E - (barrier_proto ? 1u : 2u);
        if (!wait_consumers_done(a.cflag + u.cflag0, u.ncflag, target, st, a.spin_ns)) {
          if (lane == 0) record_timeout(st, (int)W.rank, (int)it.unit, 1, E);
          failed = true;
          break;
        }
      }
      if (delay_producer && a.dbg) {
        // adversarial interleaving: stage only after the paused consumer has loaded
        if (lane == 0) {
          const uint64_t t0 = globaltimer();
          while ((int32_t)(ld_acquire_u32(a.dbg + it.unit) - E) < 0 &&
                 globaltimer() - t0 < a.inject_max_ns) {
          }
        }
        __syncwarp();
      }
      const uint32_t nvec = u.nbytes >> 4;
      char *dst = a.xbuf + (size_t)b * a.xpar + u.xoff + (size_t)it.slot * u.nbytes * slot_mult;
      uint4 x = make_uint4(0, 0, 0, 0);
      uint2 h = make_uint2(0u, 0u);
      if (pipelined) {
        x = nx;
        if (tagged && !nh_ready && lane < nvec) h = tag_part(x, lane);
      } else if constexpr (GEMV) {
        // fused producer: the CTA's compute warps have made this piece of the payload (W_r x,
        // one ordered chain per output) from the rows and the x the streamers staged
        if (!gemv_take(a, gpiece++, nvec, lane, x)) {
          if (lane == 0) record_timeout(st, (int)W.rank, (int)it.unit, 6, E);
          failed = true;
          break;
        }
        if (tagged && lane < nvec) h = tag_part(x, lane);
      } else if (lane < nvec) {
        const coll_ref_t r = a.refs[u.src0 + it.slot];
        x = ld_nc_v4(a.ptr.in[r.rank] + r.off + in_off + u.start + lane * 16);
        if (tagged) h = tag_part(x, lane);
      }
      if constexpr (LL) {
        // tagged data: every 4 payload bytes travel with the epoch in one 8-byte word
        if (lane < nvec && !skip_notify) {
          const unsigned long long ep = (unsigned long long)E << 32;
          st_relaxed_v2u64(dst + lane * 32, ep | x.x, ep | x.y);
          st_relaxed_v2u64(dst + lane * 32 + 16, ep | x.z, ep | x.w);
        }
      } else if (lane < nvec) {
        st_v4(dst + lane * 16, x);
      }
      uint2 tag = make_uint2(0u, 0u);
      if (tagged) {
        const uint2 hs = pipelined && nh_ready ? nh : reduce_add2(h);
        tag = make_uint2(tag_fold(hs.x, E), tag_fold_b(hs.y, E));
      }
      __syncwarp();
      if (lane == 0 && !skip_notify && !ll) {
        unsigned long long *fp = a.pflag + (size_t)b * a.n_pflag + u.pflag0 + it.slot;
        const unsigned long long fv = flag_word(E, tag.x, tag.y);
        if (relaxed) st_relaxed_u64(fp, fv); else st_release_u64(fp, fv);
      }
      if (pipelined) {
        nh_ready = false;
        if (i + 1 < a.n_epochs && lane < nvec) nx = ld_nc_v4(sin_base + in_off_next + lane * 16);
      }
    }
    if (failed) break;
    if (pst) a.stamps[2 + 4 * i] = globaltimer();

    // ---------------- Consume
    for (uint32_t c = W.c0; c < c_end; ++c) {
      const coll_item_t it = single_c ? cit : a.citems[c];
      const coll_unit_t u = single_c ? cu : a.units[it.unit];
      const uint32_t n = u.nsrc;
      const uint32_t nvec = u.nbytes >> 4;
      const bool active = lane < nvec;
      const char *xb = a.xbuf + (size_t)b * a.xpar + u.xoff;
      const unsigned long long *pf = a.pflag + (size_t)b * a.n_pflag + u.pflag0;
      uint4 res = make_uint4(0, 0, 0, 0);
      bool have = false;
      bool retried = false;
      if constexpr (LL) {
        // Poll the tagged words of every producer until each carries epoch E (bounded),
        // then reduce in producer order; batches of 8 producers.
        typename EngAcc<KIND>::type acc;
        const size_t pstride = (size_t)u.nbytes * 2;
        bool ok = true;
        uint32_t rounds = 0;
        for (uint32_t k0 = 0; k0 < n && ok; k0 += 8) {
          const uint32_t kn = n - k0 < 8 ? n - k0 : 8;
          uint4 d[8];
          uint32_t pending = active ? ((1u << kn) - 1u) : 0u;
          uint64_t t0 = 0;
          for (uint32_t r = 0;; ++r) {
#pragma unroll
            for (uint32_t k = 0; k < 8; ++k) {
              if (pending & (1u << k)) {
                unsigned long long w0, w1, w2, w3;
                const char *src = xb + (size_t)(k0 + k) * pstride + lane * 32;
                ld_relaxed_v2u64(src, w0, w1);
                ld_relaxed_v2u64(src + 16, w2, w3);
                if ((uint32_t)(w0 >> 32) == E && (uint32_t)(w1 >> 32) == E &&
                    (uint32_t)(w2 >> 32) == E && (uint32_t)(w3 >> 32) == E) {
                  d[k] = make_uint4((uint32_t)w0, (uint32_t)w1, (uint32_t)w2, (uint32_t)w3);
                  pending &= ~(1u << k);
                }
              }
            }
            if (__all_sync(FULL, pending == 0)) break;
            ++rounds;
            if ((r & 31u) == 31u) {
              const uint64_t now = globaltimer();
              if (t0 == 0) t0 = now;
              const bool late = (t0 != now && now - t0 > a.spin_ns) || ld_relaxed_u32(&st->abort);
              if (__any_sync(FULL, late)) {
                ok = false;
                break;
              }
            }
          }
          if (ok && active) {
#pragma unroll
            for (uint32_t k = 0; k < 8; ++k)
              if (k < kn) {
                if (k0 + k == 0) acc.init(d[k]); else acc.add(d[k]);
              }
          }
        }
        if (!ok) {
          if (lane == 0) record_timeout(st, (int)W.rank, (int)it.unit, 2, E);
          failed = true;
          break;
        }
        ++n_checks;
        if (rounds) ++n_retries;
        res = active ? acc.pack() : make_uint4(0, 0, 0, 0);
        have = true;
      }
      if (!LL && spec_proto && n <= 32) {
        // Speculative consume: load and reduce without waiting, then validate.
        unsigned long long f = 0;
        uint2 myh = make_uint2(0u, 0u);
        // (the prefetched next input is hashed while this attempt's loads are in flight)
        const bool side = pipelined && tagged && !nh_ready;
        // The speculation window: loads issued right after this warp's own notify mostly
        // race the peers' stores of the same epoch and fail validation; a short wait first
        // trades a little latency for fewer reloads.
        if (win >= 8u) spin_ns(win >> 3);
        res = spec_attempt<KIND>(xb, u.nbytes, n, lane, active, tagged, pf, !relaxed,
                                 !pause_consumer, f, myh, side, nx,
                                 pipelined ? (su.nbytes >> 4) : 0u, nh);
        if (side) nh_ready = true;
        if (pause_consumer) {
          __syncwarp();
          if (lane == 0 && a.dbg) st_release_u32(a.dbg + it.unit, E);
          spin_ns(a.inject_pause_ns);
          if (lane < n) f = relaxed ? ld_relaxed_u64(pf + lane) : ld_acquire_u64(pf + lane);
        }
        uint32_t fe = flag_epoch(f);
        bool ok;
        if (literal) {
          // the pages' reduced flag: the epochs add up to n * E (16-bit epoch fields)
          const uint32_t sum = __reduce_add_sync(FULL, lane < n ? fe : 0u);
          ok = ((sum - n * E) & 0xFFFFu) == 0u;
        } else {
          ok = tags_match(f, myh, n, E, lane);
        }
        ++n_checks;
        // adaptive window (in eighths of a ns): 1/8 ns shorter after a passed first attempt,
        // 2 ns longer after one that failed and passed at the first reload (a race with the
        // peers' stores, which a wider window avoids; a producer that is late shows as
        // several reloads instead, and a window does not help there), so that about one
        // first attempt in seventeen fails; small steps keep the window close to where it
        // balances (steps of 4 and 40 ns measured 4 % slower per epoch)
        if (a.spec_adapt && ok) win = win > 0u ? win - 1u : 0u;
        if (ok) {
          have = true;
        } else {
          ++n_retries;
          retried = true;
          if (relaxed) {
            // No ordering to lean on: reload payload and flags until the content tags
            // match (bounded by the spin limit and the abort word).
            uint64_t t0 = globaltimer();
            for (uint32_t k = 0;; ++k) {
              uint2 unused = make_uint2(0u, 0u);
              res = spec_attempt<KIND>(xb, u.nbytes, n, lane, active, true, pf, false, true, f,
                                       myh, false, nx, 0u, unused);
              fe = flag_epoch(f);
              if (tags_match(f, myh, n, E, lane)) {
                have = true;
                if (a.spec_adapt && k == 0) win = win < (1998u << 3) ? win + 16u : (2000u << 3);
                break;
              }
              const bool late = (globaltimer() - t0 > a.spin_ns) ||
                                ((k & 31u) == 31u && ld_relaxed_u32(&st->abort));
              if (__any_sync(FULL, late)) break;
            }
            if (!have) {
              if (lane == 0) record_timeout(st, (int)W.rank, (int)it.unit, 3, E);
              failed = true;
              break;
            }
          } else {
            // Lanes whose acquire already saw epoch E need no further wait; the others spin
            // until their producer notifies. Then reload everything after the acquires.
            bool wok = true;
            for (uint32_t j = lane; j < n; j += 32) {
              if (j == lane && fe == (E & 0xFFFFu)) continue;
              wok = wok && spin_u64(pf + j,
                                    [E](unsigned long long v) { return flag_is(v, E); },
                                    st, a.spin_ns);
            }
            if (!__all_sync(FULL, wok)) {
              if (lane == 0) record_timeout(st, (int)W.rank, (int)it.unit, 3, E);
              failed = true;
              break;
            }
            res = gather_pieces<KIND>(xb, u.nbytes, n, lane, active);
            have = true;
          }
        }
      }
      if (!have) {
        // Top barrier: wait until every producer of the unit has notified epoch E,
        // then load with L1-bypassing loads.
        if (!wait_producers(pf, n, E, st, a.spin_ns)) {
          if (lane == 0) record_timeout(st, (int)W.rank, (int)it.unit, retried ? 3 : 2, E);
          failed = true;
          break;
        }
        res = gather_pieces<KIND>(xb, u.nbytes, n, lane, active);
      }
      if (pst && c == W.c0) a.stamps[3 + 4 * i] = globaltimer();
      if (PULL && (u.flags & COLL_UNIT_PULL)) {
        // two-shot pull: publish the reduced piece in this parity's slot of rbuf, once
        // every consumer has pulled the piece it held before (the two-shot bottom barrier)
        const uint32_t target = E - (barrier_proto ? 1u : 2u);
        if (!wait_consumers_done(a.dflag + u.dflag0, u.ndst, target, st, a.spin_ns)) {
          if (lane == 0) record_timeout(st, (int)W.rank, (int)it.unit, 7, E);
          failed = true;
          break;
        }
        if (active) st_v4(a.rbuf + (size_t)b * a.rpar + u.roff + lane * 16, res);
        __syncwarp();
        if (lane == 0) st_release_u32(a.rflag + (size_t)b * a.n_units + it.unit, E);
      } else if (active) {
        if (it.slot == COLL_SLOT_ALL) {
          for (uint32_t d = 0; d < u.ndst; ++d) {
            const coll_ref_t r = a.refs[u.dst0 + d];
            st_v4(a.ptr.out[r.rank] + r.off + out_off + u.start + lane * 16, res);
          }
        } else if (single_c) {
          st_v4(cout_base + out_off + lane * 16, res);
        } else {
          const coll_ref_t r = a.refs[u.dst0 + it.slot];
          st_v4(a.ptr.out[r.rank] + r.off + out_off + u.start + lane * 16, res);
        }
      }
      if (barrier_proto || (u.flags & COLL_UNIT_DONE_FLAGS)) {
        __syncwarp();
        if (lane == 0)
          st_release_u32(a.cflag + u.cflag0 + (it.slot == COLL_SLOT_ALL ? 0u : it.slot), E);
      }
    }
    if (failed) break;

    // ---------------- Pull (two-shot pull): copy each owner's reduced piece of epoch E
    for (uint32_t q = W.p0; PULL && q < W.p1; ++q) {
      const coll_item_t it = a.pitems[q];
      const coll_unit_t u = a.units[it.unit];
      bool ok = true;
      if (lane == 0) ok = spin_done(a.rflag + (size_t)b * a.n_units + it.unit, E, st, a.spin_ns);
      if (!__shfl_sync(FULL, ok, 0)) {
        if (lane == 0) record_timeout(st, (int)W.rank, (int)it.unit, 8, E);
        failed = true;
        break;
      }
      __syncwarp();  // lane 0's acquire orders every lane's loads below
      if (lane < (u.nbytes >> 4)) {
        const uint4 v = ld_relaxed_v4(a.rbuf + (size_t)b * a.rpar + u.roff + lane * 16);
        const coll_ref_t r = a.refs[u.dst0 + it.slot];
        st_v4(a.ptr.out[r.rank] + r.off + out_off + u.start + lane * 16, v);
      }
      __syncwarp();
      if (lane == 0) st_release_u32(a.dflag + u.dflag0 + it.slot, E);  // read: may reuse
    }
    if (failed) break;
    if (chained) {
      __syncwarp();
      if (lane == 0) red_release_add_u32(a.rank_done + W.rank, 1u);
    }
    if (pipelined && tagged && !nh_ready && !failed) {
      nh = reduce_add2(lane < (su.nbytes >> 4) ? tag_part(nx, lane) : make_uint2(0u, 0u));
      nh_ready = true;
    }
    if (stamp && (uint32_t)i < a.stamp_cap) a.stamps[phases ? 4 + 4 * i : i + 1] = globaltimer();
  }
  if constexpr (GEMV) gemv_finish(lane);
  if (lane == 0) {
    if (n_checks) atomicAdd(&st->spec_checks, (unsigned long long)n_checks);
    if (n_retries) atomicAdd(&st->spec_retries, (unsigned long long)n_retries);
  }
}

// Flag ping-pong between block 0 and block `peer` (one thread each): block 0 stores
// ping i, block peer answers with pong i. out: [0] ns for all round trips, [1] unused,
// [2] SM of block 0, [3] SM of block peer, [4] 1 if a wait gave up.
__global__ void __launch_bounds__(32) probe_rtt_kernel(unsigned long long *flags, uint32_t iters,
                                                       uint32_t peer, unsigned long long *out,
                                                       uint64_t limit) {
  if (threadIdx.x != 0) return;
  uint32_t smid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  if (blockIdx.x == 0) {
    out[2] = smid;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1; i <= iters; ++i) {
      st_relaxed_u64(&flags[32], i);
      for (uint32_t k = 0; ld_acquire_u64(&flags[0]) != i; ++k) {
        if ((k & 63u) == 63u && globaltimer() - t0 > limit) {
          out[4] = 1;
          st_relaxed_u64(&flags[64], 1);
          return;
        }
      }
    }
    out[0] = globaltimer() - t0;
  } else if (blockIdx.x == peer) {
    out[3] = smid;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1; i <= iters; ++i) {
      for (uint32_t k = 0; ld_acquire_u64(&flags[32]) != i; ++k) {
        if ((k & 63u) == 63u && (globaltimer() - t0 > limit || ld_relaxed_u64(&flags[64]))) {
          out[4] = 1;
          return;
        }
      }
      st_relaxed_u64(&flags[0], i);
    }
  }
}

int kind_of(int op, int dtype) {
  if (op == COLL_OP_COPY) return 0;
  return dtype == COLL_BF16 ? 1 : 2;
}

}  // namespace

cudaError_t launch_zero_copy(int op, int dtype, int keep, const ZcArgs &a, int ctas,
                             cudaStream_t s) {
  const int kind = kind_of(op, dtype);
  const uint64_t total = (uint64_t)a.ntiles * a.n_epochs;
  if (total == 0) return cudaSuccess;
  const uint64_t need = (total + 7) / 8;  // 8 warps per CTA
  const int grid = (int)((uint64_t)ctas < need ? (uint64_t)ctas : need);
  const void *fn;
  if (a.tree && kind != 0) {
    switch (kind * 2 + (keep ? 1 : 0)) {
      case 2: fn = (const void *)zc_kernel<1, false, true>; break;
      case 3: fn = (const void *)zc_kernel<1, true, true>; break;
      case 4: fn = (const void *)zc_kernel<2, false, true>; break;
      default: fn = (const void *)zc_kernel<2, true, true>; break;
    }
  } else {
    switch (kind * 2 + (keep ? 1 : 0)) {
      case 0: fn = (const void *)zc_kernel<0, false, false>; break;
      case 1: fn = (const void *)zc_kernel<0, true, false>; break;
      case 2: fn = (const void *)zc_kernel<1, false, false>; break;
      case 3: fn = (const void *)zc_kernel<1, true, false>; break;
      case 4: fn = (const void *)zc_kernel<2, false, false>; break;
      default: fn = (const void *)zc_kernel<2, true, false>; break;
    }
  }
  ZcArgs la = a;
  void *args[] = {(void *)&la};
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

static const void *engine_fn(int kind, bool gemv, bool ll, bool pull, int fp = 0) {
  if (gemv) return pull ? (const void *)engine_kernel<1, true, false, true, 0>
                        : (const void *)engine_kernel<1, true, false, false, 0>;
  if (ll) {
    switch (kind) {
      case 0: return (const void *)engine_kernel<0, false, true, false, 0>;
      case 1: return (const void *)engine_kernel<1, false, true, false, 0>;
      default: return (const void *)engine_kernel<2, false, true, false, 0>;
    }
  }
  if (pull && kind != 0)  // (pull plans are sums)
    return kind == 1 ? (const void *)engine_kernel<1, false, false, true, 0>
                     : (const void *)engine_kernel<2, false, false, true, 0>;
  if (fp != 0 && kind != 0) {  // (the specialised variants are sums)
    switch ((kind - 1) * 6 + fp) {
      case 1: return (const void *)engine_kernel<1, false, false, false, 1>;
      case 2: return (const void *)engine_kernel<1, false, false, false, 2>;
      case 3: return (const void *)engine_kernel<1, false, false, false, 3>;
      case 4: return (const void *)engine_kernel<1, false, false, false, 4>;
      case 5: return (const void *)engine_kernel<1, false, false, false, 5>;
      case 6: return (const void *)engine_kernel<1, false, false, false, 6>;
      case 7: return (const void *)engine_kernel<2, false, false, false, 1>;
      case 8: return (const void *)engine_kernel<2, false, false, false, 2>;
      case 9: return (const void *)engine_kernel<2, false, false, false, 3>;
      case 10: return (const void *)engine_kernel<2, false, false, false, 4>;
      case 11: return (const void *)engine_kernel<2, false, false, false, 5>;
      default: return (const void *)engine_kernel<2, false, false, false, 6>;
    }
  }
  switch (kind) {
    case 0: return (const void *)engine_kernel<0, false, false, false, 0>;
    case 1: return (const void *)engine_kernel<1, false, false, false, 0>;
    default: return (const void *)engine_kernel<2, false, false, false, 0>;
  }
}

// The specialised variant a run of these arguments may use (0: the general engine).
// FP 1/2: tagged / fence-free check; 3/4: the same with one stamp per epoch; 5/6: the same
// checks with chained epochs (no stamps).
static int engine_fp(int kind, const EngArgs &a) {
  if (kind == 0 || a.gemv_k != 0 || a.rpar != 0 || !a.single_items || a.inject_flags != 0 ||
      (a.stamps != nullptr && a.stamp_phases) || a.dbg != nullptr)
    return 0;
  const bool chain = a.chain && a.rank_done;
  if (chain && a.stamps != nullptr) return 0;
  const int off = chain ? 4 : a.stamps != nullptr ? 2 : 0;
  if (a.protocol == COLL_PROTO_SPEC && a.spec_check == COLL_SPEC_TAGGED) return 1 + off;
  if (a.protocol == COLL_PROTO_SPEC && a.spec_check == COLL_SPEC_TAGGED_RELAXED) return 2 + off;
  return 0;
}

cudaError_t engine_max_coresident(int op, int dtype, int protocol, int datapath, int *max_ctas) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int kind = kind_of(op, dtype);
  const bool ll = protocol == COLL_PROTO_LL, pull = datapath == COLL_DP_TWOSHOT_PULL;
  // a run may use a specialised variant: every variant it may use must fit
  int per_sm = 1 << 30;
  for (int fp = 0; fp <= ((kind != 0 && !ll && !pull) ? 6 : 0); ++fp) {
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, engine_fn(kind, false, ll, pull, fp),
                                                      32, 0);
    if (e != cudaSuccess) return e;
    per_sm = n < per_sm ? n : per_sm;
  }
  *max_ctas = per_sm * sms;
  return cudaSuccess;
}

uint32_t gemv_ring_slots(uint32_t pitch) {
  const uint32_t n = kGemvRingBytes / (kGemvRows * pitch);
  return n < kGemvMaxSlots ? n : kGemvMaxSlots;
}

cudaError_t engine_gemv_max_coresident(bool pull, int *max_ctas) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const void *fn = engine_fn(1, true, false, pull);
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemvSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kGemvThreads, kGemvSmemBytes);
  if (e != cudaSuccess) return e;
  *max_ctas = per_sm * sms;
  return cudaSuccess;
}

cudaError_t launch_probe_rtt(unsigned long long *flags, uint32_t iters, uint32_t peer,
                             unsigned long long *out, uint64_t limit, cudaStream_t s) {
  void *args[] = {(void *)&flags, (void *)&iters, (void *)&peer, (void *)&out, (void *)&limit};
  return cudaLaunchCooperativeKernel((const void *)probe_rtt_kernel, dim3(peer + 1), dim3(32),
                                     args, 0, s);
}

cudaError_t launch_engine(int op, int dtype, const EngArgs &a, const GemvMaps *maps,
                          cudaStream_t s) {
  if (a.nwarps == 0 || a.n_epochs == 0) return cudaSuccess;
  const bool gemv = a.gemv_k != 0;
  if (gemv && !maps) return cudaErrorInvalidValue;
  NoMaps none{0};
  void *args[] = {(void *)&a, gemv ? (void *)maps : (void *)&none};
  const int kind = kind_of(op, dtype);
  const void *fn =
      engine_fn(kind, gemv, a.protocol == COLL_PROTO_LL, a.rpar != 0, engine_fp(kind, a));
  if (gemv) {
    // (once per variant: the attribute stays set, and a stream capture then records the
    // launch alone)
    static bool smem_set[64][2] = {};
    int dev = 0;
    const cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess) return de;
    bool scratch = false;
    bool &set = dev >= 0 && dev < 64 ? smem_set[dev][a.rpar != 0 ? 1 : 0] : scratch;
    if (!set) {
      const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)kGemvSmemBytes);
      if (e != cudaSuccess) return e;
      set = true;
    }
  }
  return cudaLaunchCooperativeKernel(fn, dim3(a.nwarps), dim3(gemv ? kGemvThreads : 32), args,
                                     gemv ? kGemvSmemBytes : 0, s);
}

}  // namespace coll
