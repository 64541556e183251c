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
// path (same arithmetic, same order).
template <int KIND, bool KEEP, bool TREE>
__global__ void __launch_bounds__(256, TREE ? 2 : 3) zc_kernel(const ZcArgs a) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint64_t gw = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint64_t nw = ((uint64_t)gridDim.x * blockDim.x) >> 5;
  const uint64_t total = (uint64_t)a.ntiles * a.n_epochs;
  constexpr uint64_t kOffMask = (1ull << 56) - 1u;
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
// The fused-producer variant runs twelve warps per CTA in three warpgroups. Warp 0 plays the
// engine warp; warps 4..11 are compute warps: at each stage compute warp b computes k-block b
// of the piece's dot products (lane l: outputs 8l..8l+7). Block b covers rows
// [b*k/8, (b+1)*k/8): products rounded to binary32, added in row order from the block's
// first product; warp 0 then adds the eight block sums in block order and rounds once to
// bf16. Warps 1..3 only complete the first warpgroup. The register file is split by
// warpgroup (setmaxnreg): the engine's warpgroup takes 248 registers a thread, the compute
// warpgroups 120, so neither the engine state nor the compute loop spills.
//
// The weight rows reach the compute warps through shared-memory slots of 16 rows, each
// filled by one tensor copy (TMA: a box of 256 columns x 16 rows of W_r, so a ragged last
// piece reads zeros past the matrix); each compute warp owns 3 slots (a private ring) and
// streams its own k-block through them. Fill q of warp b (its q-th slot of rows over the run:
// piece q / (k/128), slot q % (k/128) of block b, pieces in epoch-major stage-item order)
// lands in the warp's slot q % 3; having read fill q, the warp issues fill q + 3 into the
// same slot. So each warp always has its next 3 slots (48 rows) in flight: while the engine
// warp runs the exchange of one epoch, the next piece's rows are already arriving (the
// weights do not depend on the epoch's data). Few large fills beat many small ones here:
// streaming rows through shared memory is bound by its bandwidth (every byte is written by
// the copy and read once), and each fill costs a fixed wait and issue on top.
constexpr uint32_t kGemvWarps = 8;                                   // compute warps
constexpr uint32_t kGemvFirst = 4;                                   // warp of compute warp 0
constexpr uint32_t kGemvThreads = 32 * (kGemvFirst + kGemvWarps);   // 384
constexpr uint32_t kGemvBarThreads = 32 * (1 + kGemvWarps);          // engine + compute warps
constexpr uint32_t kGemvLaunchRegs = 168;  // per thread at launch: 65536 / 384, rounded to 8
constexpr uint32_t kGemvEngineRegs = 248;  // engine warpgroup after the split
constexpr uint32_t kGemvComputeRegs = 120; // compute warpgroups after the split
static_assert(128 * kGemvEngineRegs + 256 * kGemvComputeRegs <= kGemvThreads * kGemvLaunchRegs,
              "the split must fit in the registers the CTA was launched with");
constexpr uint32_t kGemvRows = 16;                       // weight rows per ring slot (one copy)
constexpr uint32_t kGemvCols = 256;                      // bf16 columns per copied row (a piece)
constexpr uint32_t kGemvPitch = 2 * kGemvCols;           // bytes per staged row
constexpr uint32_t kGemvSlotBytes = kGemvRows * kGemvPitch;
constexpr uint32_t kGemvSlotsPerWarp = 3;
constexpr uint32_t kGemvSlots = kGemvSlotsPerWarp * kGemvWarps;  // 192 KiB of rows in flight
// (the ring starts 128-byte aligned: the tensor copies land there)
constexpr uint32_t kGemvSmemBytes = kGemvSlots * kGemvSlotBytes + kGemvSlots * 8 + 128;
constexpr uint32_t kGemvMaxItems = 16;                   // stage items whose rows are cached

struct GemvShared {
  const char *xp;    // x vector of this epoch
  uint32_t active;   // lanes below this hold outputs
  uint32_t exit;     // set by warp 0: the other warps return
  uint32_t fail;     // a compute warp's ring wait gave up
  uint32_t nitems;   // stage items of this warp, in order
  uint32_t S;        // slots per piece
  uint64_t total;    // fills of the whole run, per compute warp
  const CUtensorMap *maps;                 // W_r of each rank (kernel parameters)
  const CUtensorMap *wmap[kGemvMaxItems];  // each cached item's matrix ...
  uint32_t wcol[kGemvMaxItems];            // ... and its first column
  uint32_t fills[kGemvSlots];              // fills issued per slot
  float part[kGemvWarps][32][8];
};

__device__ __forceinline__ GemvShared &gemv_smem() {
  __shared__ GemvShared g;
  return g;
}

struct GemvRing {
  unsigned char *rows;  // [kGemvSlots][kGemvRows][kGemvPitch]
  uint64_t *full;       // [kGemvSlots] completes when a fill's rows have landed
};

__device__ __forceinline__ GemvRing gemv_ring() {
  extern __shared__ __align__(128) unsigned char gemv_dyn[];
  GemvRing r;
  r.rows = gemv_dyn + ((128u - (smem_u32(gemv_dyn) & 127u)) & 127u);
  r.full = reinterpret_cast<uint64_t *>(r.rows + kGemvSlots * kGemvSlotBytes);
  return r;
}

__device__ __forceinline__ void gemv_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kGemvBarThreads) : "memory");
}

// Where the rows of one fill come from: W_r's tensor map and the piece's first column.
struct GemvSrc {
  const CUtensorMap *map;
  uint32_t col;
};

// Rows of item `idx` of this CTA's warp: cached in shared memory for the first items, read
// from the plan tables beyond that.
__device__ __forceinline__ GemvSrc gemv_item(const EngArgs &a, const GemvShared &g,
                                             const coll_warp_t &W, uint32_t idx) {
  if (idx < kGemvMaxItems) return GemvSrc{g.wmap[idx], g.wcol[idx]};
  const coll_item_t it = a.sitems[W.s0 + idx];
  const coll_unit_t u = a.units[it.unit];
  const coll_ref_t r = a.refs[u.src0 + it.slot];
  return GemvSrc{g.maps + r.rank, (uint32_t)((r.off + u.start) >> 1)};
}

// Issue one fill into `slot` (all lanes call; lane 0 issues): rows 16*rj..16*rj+15 of the
// piece's 256 columns, one tensor copy whose bytes complete the slot's barrier. Lane 0
// counts the fill. The slot must be free: every lane of the calling warp has finished its
// reads of the previous fill (their values are in registers and the warp has synchronised).
__device__ __forceinline__ void gemv_fill(GemvShared &g, const GemvRing &ring, uint32_t slot,
                                          const GemvSrc &src, uint32_t rj, uint32_t lane) {
  if (lane == 0) {
    *reinterpret_cast<volatile uint32_t *>(&g.fills[slot]) = g.fills[slot] + 1u;
    mbar_expect_tx(&ring.full[slot], kGemvSlotBytes);
    tensor_load_2d(ring.rows + slot * kGemvSlotBytes, src.map, src.col, rj * kGemvRows,
                   &ring.full[slot]);
  }
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
// bf16 elements 2j, 2j+1 of a word -> {binary32, binary32}
__device__ __forceinline__ uint64_t bf16x2_widen(uint32_t w) {
  return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Eight rows of this lane's eight outputs: acc[p] holds outputs (2p, 2p+1).
template <bool FIRST>
__device__ __forceinline__ void gemv_rows8(uint64_t acc[4], const uint4 w[8], uint4 xv) {
  const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
  for (uint32_t t = 0; t < 8; ++t) {
    const float xf = __uint_as_float((t & 1u) ? (xw[t >> 1] & 0xFFFF0000u) : (xw[t >> 1] << 16));
    const uint64_t xx = f2_pack(xf, xf);
    const uint32_t ww[4] = {w[t].x, w[t].y, w[t].z, w[t].w};
#pragma unroll
    for (uint32_t p = 0; p < 4; ++p) {
      const uint64_t prod = f2_mul(bf16x2_widen(ww[p]), xx);
      acc[p] = (FIRST && t == 0) ? prod : f2_add(acc[p], prod);
    }
  }
}

// Position of a compute warp's reads in its private ring, and of the refills it issues. It
// lives across blocks and only ever steps forward (no division on the compute path).
struct GemvCursor {
  uint64_t q, lap;  // fill read next: number q, lap q / 3 of the warp's slot q % 3
  uint32_t slot;    // ring slot (warp base + q % 3)
  uint32_t rp_j;    // refill q + 3: slot rp_j of the block ...
  uint32_t ri;      // ... of stage item ri
  GemvSrc src;      // rows of item ri
};

// Refills of the next piece's slots, held back until the block's results are handed over:
// n consecutive fills (consecutive slots of the ring, consecutive refill positions), the
// first of them into `slot`, slot rj of the block of stage item ri.
struct GemvPending {
  uint32_t n, slot, rj, ri;
  GemvSrc src;
};

// Compute warp `wid`, before its first block: issue its first 3 fills and set the cursor
// (next read: fill 0; next refill: fill 3).
__device__ void gemv_warp_prologue(const EngArgs &a, GemvShared &g, const GemvRing &ring,
                                   const coll_warp_t &W, uint32_t wid, uint32_t lane,
                                   GemvCursor &c) {
  const uint32_t bs = g.S / kGemvWarps;
  uint32_t j = 0, ri = 0;
  GemvSrc src = gemv_item(a, g, W, 0);
  for (uint32_t q = 0; q < kGemvSlotsPerWarp; ++q) {
    if (q < g.total) gemv_fill(g, ring, wid * kGemvSlotsPerWarp + q, src, wid * bs + j, lane);
    if (++j == bs) {
      j = 0;
      if (++ri == g.nitems) ri = 0;
      src = gemv_item(a, g, W, ri);
    }
  }
  c.q = 0;
  c.lap = 0;
  c.slot = wid * kGemvSlotsPerWarp;
  c.rp_j = j;
  c.ri = ri;
  c.src = src;
}

// This warp's k-block of piece `piece` into g.part[wid][lane], streaming the block's rows
// through the warp's private ring (see above). The readiness of the slots already issued is
// tested at once, so slots that landed during the exchange cost no wait each.
__device__ __forceinline__ void gemv_block(const EngArgs &a, GemvShared &g, const GemvRing &ring,
                                           const coll_warp_t &W, uint32_t wid, uint32_t lane,
                                           GemvCursor &c, GemvPending &pend) {
  const uint32_t bs = g.S / kGemvWarps;  // slots per block
  const uint64_t total = g.total;
  const uint32_t base = wid * kGemvSlotsPerWarp;
  const bool act = lane < g.active;
  // x of this block: lane t holds the 16 values of slot 32c+t of chunk c, loaded together
  // (one memory round trip per 32 slots), and each slot's values are broadcast by shuffle
  const char *xp = g.xp + (size_t)wid * bs * (kGemvRows * 2);
  uint64_t acc[4] = {0, 0, 0, 0};
  uint4 xl[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
  uint32_t ready = 0;  // bit t: the fill of slot 32c+t of this chunk has already landed
  const uint64_t qe = c.q + bs;  // first fill of the next piece
  pend.n = 0;
  bool done = true;
  for (uint32_t j = 0; j < bs; ++j) {
    if ((j & 31u) == 0u) {
      // per chunk of 32 slots: one x load and one readiness test per lane, in parallel
      // (only the fills already issued, at most 3 ahead, can have landed)
      bool r = false;
      if (j + lane < bs) {
        xl[0] = ld_nc_v4(xp + (size_t)(j + lane) * 32);
        xl[1] = ld_nc_v4(xp + (size_t)(j + lane) * 32 + 16);
      }
      if (j + lane < bs && lane < kGemvSlotsPerWarp) {
        const uint32_t o = c.slot - base + lane;  // fill c.q + lane: slot o % 3, lap + o / 3
        const uint32_t wrap = o >= kGemvSlotsPerWarp ? 1u : 0u;
        r = mbar_test_wait(&ring.full[base + o - wrap * kGemvSlotsPerWarp],
                           (uint32_t)((c.lap + wrap) & 1u));
      }
      ready = __ballot_sync(FULL, r);
      __syncwarp();  // orders each lane's acquiring test before every lane's reads
    }
    bool ok = true;
    if (!((ready >> (j & 31u)) & 1u)) {
      // (this warp issued the fill itself, so the slot's previous phase has completed and
      // the parity identifies the fill)
      if (lane == 0)
        ok = mbar_wait_until(&ring.full[c.slot], (uint32_t)(c.lap & 1u), a.spin_ns,
                             [&a]() { return ld_relaxed_u32(&a.st->abort) != 0u; });
      ok = __shfl_sync(FULL, ok, 0);
      __syncwarp();  // orders lane 0's acquiring wait before every lane's reads
    }
    if (!ok) {
      if (lane == 0) {
        record_timeout(a.st, (int)W.rank, -1, 6, 0);
        g.fail = 1;
      }
      done = false;
      break;
    }
    const unsigned char *s = ring.rows + c.slot * kGemvSlotBytes + lane * 16;
#pragma unroll
    for (uint32_t h = 0; h < 2; ++h) {  // rows 8h..8h+7 of the slot
      uint4 xv;
      xv.x = __shfl_sync(FULL, xl[h].x, j & 31u);
      xv.y = __shfl_sync(FULL, xl[h].y, j & 31u);
      xv.z = __shfl_sync(FULL, xl[h].z, j & 31u);
      xv.w = __shfl_sync(FULL, xl[h].w, j & 31u);
      uint4 w[8];
#pragma unroll
      for (uint32_t t = 0; t < 8; ++t)
        w[t] = act ? *reinterpret_cast<const uint4 *>(s + (8 * h + t) * kGemvPitch)
                   : make_uint4(0, 0, 0, 0);
      if (j == 0 && h == 0) gemv_rows8<true>(acc, w, xv); else gemv_rows8<false>(acc, w, xv);
    }
    // The slot's rows are in registers and used: once the warp has synchronised, the copy
    // may overwrite the slot. A refill this block still needs is issued now; refills for
    // later pieces wait for the end of the block, so that their copies stream during the
    // exchange instead of competing with this block's.
    __syncwarp();
    if (c.q + kGemvSlotsPerWarp < total) {
      if (c.q + kGemvSlotsPerWarp < qe) {
        gemv_fill(g, ring, c.slot, c.src, wid * bs + c.rp_j, lane);
      } else {
        if (pend.n == 0) {
          pend.slot = c.slot;
          pend.rj = c.rp_j;
          pend.ri = c.ri;
          pend.src = c.src;
        }
        ++pend.n;
      }
    }
    ++c.q;
    if (++c.slot == base + kGemvSlotsPerWarp) {
      c.slot = base;
      ++c.lap;
    }
    if (++c.rp_j == bs) {
      c.rp_j = 0;
      if (++c.ri == g.nitems) c.ri = 0;
      c.src = gemv_item(a, g, W, c.ri);
    }
  }
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(acc[p]));
    g.part[wid][lane][2 * p] = lo;
    g.part[wid][lane][2 * p + 1] = hi;
  }
  if (!done && lane == 0) g.fail = 1;
}

// Warp 0, before the epoch loop: cache the stage items' row sources and the run's sizes.
__device__ void gemv_prologue(const EngArgs &a, const CUtensorMap *maps, const coll_warp_t &W,
                              uint32_t lane) {
  GemvShared &g = gemv_smem();
  const uint32_t nitems = W.s1 - W.s0;
  if (lane == 0) {
    g.nitems = nitems;
    g.S = a.gemv_k / kGemvRows;
    g.total = (uint64_t)a.n_epochs * nitems * (a.gemv_k / (kGemvRows * kGemvWarps));
    g.maps = maps;
  }
  for (uint32_t idx = lane; idx < nitems && idx < kGemvMaxItems; idx += 32) {
    const coll_item_t it = a.sitems[W.s0 + idx];
    const coll_unit_t u = a.units[it.unit];
    const coll_ref_t r = a.refs[u.src0 + it.slot];
    g.wmap[idx] = maps + r.rank;
    g.wcol[idx] = (uint32_t)((r.off + u.start) >> 1);
  }
}

// Compute warp `wid` (0..7): compute block wid whenever warp 0 opens a stage, until told to
// exit. After each block, the refills it held back are issued: their copies stream while
// warp 0 runs the exchange.
__device__ void gemv_helper_loop(const EngArgs &a, const coll_warp_t &W, uint32_t wid,
                                 uint32_t lane) {
  GemvShared &g = gemv_smem();
  const GemvRing ring = gemv_ring();
  GemvCursor c;
  GemvPending pend;
  gemv_warp_prologue(a, g, ring, W, wid, lane, c);
  for (;;) {
    gemv_bar();
    if (g.exit) return;
    gemv_block(a, g, ring, W, wid, lane, c, pend);
    gemv_bar();
    if (g.fail) continue;
    const uint32_t bs = g.S / kGemvWarps;
    const uint32_t base = wid * kGemvSlotsPerWarp;
    for (uint32_t d = 0; d < pend.n; ++d) {
      gemv_fill(g, ring, pend.slot, pend.src, wid * bs + pend.rj, lane);
      if (++pend.slot == base + kGemvSlotsPerWarp) pend.slot = base;
      if (++pend.rj == bs) {
        pend.rj = 0;
        if (++pend.ri == g.nitems) pend.ri = 0;
        pend.src = gemv_item(a, g, W, pend.ri);
      }
    }
  }
}

// Warp 0 (all 32 lanes): piece number `piece` of y = W x for the lanes below `active`;
// false if a ring wait gave up (the status word then holds the timeout).
__device__ __forceinline__ bool gemv_piece_mw(const EngArgs &a, const coll_warp_t &W,
                                              const char *xp, uint32_t active, uint64_t piece,
                                              uint32_t lane, uint4 &res) {
  GemvShared &g = gemv_smem();
  const GemvRing ring = gemv_ring();
  if (lane == 0) {
    g.xp = xp;
    g.active = active;
  }
  __syncwarp();
  gemv_bar();  // open: the compute warps start their blocks
  gemv_bar();  // every block sum is in shared memory
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = g.part[0][lane][e];
#pragma unroll
  for (uint32_t b = 1; b < kGemvWarps; ++b)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], g.part[b][lane][e]);
  res = bf16x8_pack(acc);
  return __shfl_sync(FULL, g.fail, 0) == 0u;
}

// Warp 0 at the end: release the other warps, then wait (bounded) for every fill issued
// so far, so that no bulk copy lands after the CTA has exited (after a failure some
// fills are never read).
__device__ __forceinline__ void gemv_finish(uint32_t lane) {
  GemvShared &g = gemv_smem();
  const GemvRing ring = gemv_ring();
  if (lane == 0) *reinterpret_cast<volatile uint32_t *>(&g.exit) = 1u;
  __syncwarp();
  gemv_bar();
  if (lane == 0) {
    for (uint32_t s = 0; s < kGemvSlots; ++s) {
      const uint32_t n = g.fills[s];
      if (n) mbar_wait_until(&ring.full[s], (n - 1u) & 1u, 100000000ull, []() { return false; });
    }
  }
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
// stage item and one consume item, run without fault injection, stamps or chained epochs,
// under one speculative protocol known at compile time (1 with content tags, 2 the same
// fence-free). On the single warp that carries a piece through an epoch, every runtime mode
// test is a dependent instruction on the critical path; compiled out, the decode epoch
// drops by about a sixth. (A dual-buffer variant measured slower than the general engine
// and is not built.)
// (the fused producer also takes the tensor maps of the ranks' weight matrices)
template <bool GEMV> struct MapsArg { using type = NoMaps; };
template <> struct MapsArg<true> { using type = GemvMaps; };

template <int KIND, bool GEMV, bool LL, bool PULL, int FP>
__global__ void __launch_bounds__(GEMV ? kGemvThreads : 32, 1)
    engine_kernel(const EngArgs a, const __grid_constant__ typename MapsArg<GEMV>::type maps) {
  static_assert(FP == 0 || (!GEMV && !LL && !PULL), "the specialised variants are plain");
  constexpr bool fast = FP != 0;
  const uint32_t gw = blockIdx.x;
  const uint32_t lane = threadIdx.x & 31u;
  if constexpr (GEMV) {
    const uint32_t wid = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
      GemvShared &g = gemv_smem();
      const GemvRing ring = gemv_ring();
      g.exit = 0;
      g.fail = 0;
      for (uint32_t s = 0; s < kGemvSlots; ++s) {
        g.fills[s] = 0;
        mbar_init(&ring.full[s], 1);  // the filling lane's arrival, plus the copy's bytes
      }
      mbar_init_fence();
    }
    __syncthreads();
    if (gw >= a.nwarps) return;  // (every CTA of a launch is a plan warp)
    if (wid == 0) gemv_prologue(a, maps.m, a.warps[gw], lane);
    __syncthreads();  // the item cache and the run's fill count are set
    // The register split: the compute warpgroups shrink, the engine's warpgroup grows. Each
    // role then runs to the end without rejoining the other, so that each is compiled for
    // its own register budget.
    if (wid >= kGemvFirst) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kGemvComputeRegs));
      gemv_helper_loop(a, a.warps[gw], wid - kGemvFirst, lane);
      return;
    }
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kGemvEngineRegs));
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
  const bool relaxed = fast ? FP == 2 : spec_proto && a.spec_check == COLL_SPEC_TAGGED_RELAXED;
  const bool tagged = spec_proto && !literal;
  const bool skip_notify = !fast && (a.inject_flags & COLL_INJECT_SKIP_NOTIFY) &&
                           (int)W.rank == a.inject_rank;
  const bool pause_consumer = !fast && (a.inject_flags & COLL_INJECT_SPEC_PAUSE) &&
                              (int)W.rank == a.inject_rank;
  const bool delay_producer = !fast && (a.inject_flags & COLL_INJECT_SPEC_PAUSE) &&
                              (int)W.rank == (a.inject_rank + 1) % a.R;
  const bool chained = !fast && a.chain && a.rank_done;
  const bool stagger = !fast && (a.inject_flags & COLL_INJECT_STAGGER);
  uint32_t n_checks = 0, n_retries = 0;
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
  const bool stamp = !fast && gw == 0 && lane == 0 && a.stamps;
  const bool phases = stamp && a.stamp_phases;
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
        // fused producer: the CTA's eight compute warps make this piece of the payload from
        // the weight rows the streaming warp has staged
        const coll_ref_t r = single_s ? sref : a.refs[u.src0 + it.slot];
        if (!gemv_piece_mw(a, W, a.ptr.in[r.rank] + in_off, nvec, gpiece++, lane, x)) {
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
  const dim3 block(256);
  if (a.tree && kind != 0) {
    switch (kind * 2 + (keep ? 1 : 0)) {
      case 2: zc_kernel<1, false, true><<<grid, block, 0, s>>>(a); break;
      case 3: zc_kernel<1, true, true><<<grid, block, 0, s>>>(a); break;
      case 4: zc_kernel<2, false, true><<<grid, block, 0, s>>>(a); break;
      default: zc_kernel<2, true, true><<<grid, block, 0, s>>>(a); break;
    }
    return cudaGetLastError();
  }
  switch (kind * 2 + (keep ? 1 : 0)) {
    case 0: zc_kernel<0, false, false><<<grid, block, 0, s>>>(a); break;
    case 1: zc_kernel<0, true, false><<<grid, block, 0, s>>>(a); break;
    case 2: zc_kernel<1, false, false><<<grid, block, 0, s>>>(a); break;
    case 3: zc_kernel<1, true, false><<<grid, block, 0, s>>>(a); break;
    case 4: zc_kernel<2, false, false><<<grid, block, 0, s>>>(a); break;
    default: zc_kernel<2, true, false><<<grid, block, 0, s>>>(a); break;
  }
  return cudaGetLastError();
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
    switch ((kind - 1) * 2 + fp) {
      case 1: return (const void *)engine_kernel<1, false, false, false, 1>;
      case 2: return (const void *)engine_kernel<1, false, false, false, 2>;
      case 3: return (const void *)engine_kernel<2, false, false, false, 1>;
      default: return (const void *)engine_kernel<2, false, false, false, 2>;
    }
  }
  switch (kind) {
    case 0: return (const void *)engine_kernel<0, false, false, false, 0>;
    case 1: return (const void *)engine_kernel<1, false, false, false, 0>;
    default: return (const void *)engine_kernel<2, false, false, false, 0>;
  }
}

// The specialised variant a run of these arguments may use (0: the general engine).
static int engine_fp(int kind, const EngArgs &a) {
  if (kind == 0 || a.gemv_k != 0 || a.rpar != 0 || !a.single_items || a.inject_flags != 0 ||
      a.stamps != nullptr || a.dbg != nullptr || (a.chain && a.rank_done))
    return 0;
  if (a.protocol == COLL_PROTO_SPEC && a.spec_check == COLL_SPEC_TAGGED) return 1;
  if (a.protocol == COLL_PROTO_SPEC && a.spec_check == COLL_SPEC_TAGGED_RELAXED) return 2;
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
  for (int fp = 0; fp <= ((kind != 0 && !ll && !pull) ? 2 : 0); ++fp) {
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, engine_fn(kind, false, ll, pull, fp),
                                                      32, 0);
    if (e != cudaSuccess) return e;
    per_sm = n < per_sm ? n : per_sm;
  }
  *max_ctas = per_sm * sms;
  return cudaSuccess;
}

cudaError_t engine_gemv_max_coresident(bool pull, int *max_ctas) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const void *fn = engine_fn(1, true, false, pull);
  // the in-kernel register split assumes the launch allocation it was written for
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, fn);
  if (e != cudaSuccess) return e;
  if ((uint32_t)fa.numRegs != kGemvLaunchRegs) return cudaErrorInvalidConfiguration;
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
