// Zero-copy datapath, bulk-copy (TMA) variant for large 16-byte-aligned plans, sm_103a.
//
// One persistent CTA per SM. Warps 0 and 1 are the producers: for each tile one of them
// issues one cp.async.bulk (global -> shared, completion on an mbarrier) per producer segment
// into a ring of shared-memory stages. Warps 2..9 are consumers: they wait for a stage, reduce the
// staged pieces in the plan's order (binary32, one RNE to bf16) or take the single piece
// (copy), store the result to every destination with streaming 16-byte stores, and release
// the stage. The ring keeps up to `stages` tiles of loads in flight per SM independently of
// register pressure, which is what a streaming copy/reduce needs to reach HBM bandwidth.
//
// The ring is launched as a programmatic dependent of the previous kernel in its stream: a
// CTA initialises its barriers and resolves its first batch of tile records, which are the
// plan's and never written by a run, while the previous kernel finishes, and its producer
// waits for that kernel's completion (griddep_wait) before it touches the plan's counters or
// any caller buffer. Once a CTA's producer has issued its last tile, the CTA lets the next
// kernel start (on the SMs this grid releases).
//
// Every mbarrier wait is bounded by the plan's spin limit; on expiry the CTA records
// COLL_ETIMEDOUT in the plan status, waits (bounded) for the bulk copies it issued, and
// returns.
#include <cuda_runtime.h>
#include <stdint.h>

#include "atom.cuh"
#include "engine.cuh"
#include "tma.cuh"

namespace coll {

namespace {

constexpr uint32_t kConsumerWarps = 8;
constexpr uint32_t kProducerWarps = 2;  // warps issuing copies: tile k by warp k % 2
static_assert(kProducerWarps == 2, "the issue loop and the abort path split tiles by parity");
constexpr unsigned FULLW = 0xFFFFFFFFu;
constexpr uint32_t kThreads = 32 * (kConsumerWarps + kProducerWarps);
constexpr uint32_t kClaim = 2;   // tiles per claim of the dynamic tail (the least, if guided)
constexpr uint32_t kTable = 64;  // resolved tiles held (>= 32 + the ring's stages)

// A resolved tile: its sources and destinations as pointers, sizes and counts. Producer
// warp 0 resolves a batch of tiles (one per lane) into a table of kTable entries in shared
// memory, the tile this CTA issues k-th into entry k % kTable; a stage records which entry
// it holds. Entry k % kTable was last used by tile k - kTable. Both producer warps have
// issued every tile of a batch before the next batch is written, and issuing tile k - 1
// waited for tile k - 1 - S to be released (S <= 12 stages): a batch of up to 32 tiles
// starting at k only overwrites entries of released tiles.
struct TileRec {
  const char *src[COLL_BULK_MAX_SRC];
  char *dst[COLL_BULK_MAX_DST];
  uint32_t nbytes, nsrc, ndst, pad;
};

__device__ void bulk_timeout(coll_dev_status_t *st, uint32_t tile) {
  if (atomicCAS(&st->status, 0, COLL_ETIMEDOUT) == 0) {
    st->fail_rank = -1;
    st->fail_unit = (int)tile;
    st->fail_where = 5;
    st->fail_epoch = 0;
  }
}

// KIND: 0 copy, 1 sum of bf16, 2 sum of f32.
template <int KIND, bool TREE>
__global__ void __launch_bounds__(kThreads, 1) bulk_kernel(const ZcArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ TileRec table[kTable];
  __shared__ volatile uint32_t s_abort;
  __shared__ uint32_t s_issued[kProducerWarps];  // per producer warp: 1 + its last tile issued
  __shared__ volatile uint32_t s_batch;          // tiles of the batch warp 0 has published
  __shared__ volatile uint32_t s_final;          // tiles this CTA issues in all, once known
  const uint32_t S = a.stages;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *empty = full + S;
  uint32_t *stile = reinterpret_cast<uint32_t *>(empty + S);  // table entry of each stage
  const uint32_t head = ((16u * S + 4u * S) + 127u) & ~127u;
  unsigned char *data = smem + head;
  const uint32_t stage_bytes = a.maxsrc * a.slot_bytes;
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
  const uint64_t total = (uint64_t)a.ntiles * a.n_epochs;

  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    s_abort = 0;
    for (uint32_t p = 0; p < kProducerWarps; ++p) s_issued[p] = 0;
    s_batch = 0;
    s_final = 0xFFFFFFFFu;
    mbar_init_fence();
  }
  __syncthreads();

  uint32_t consumed = 0;
  if (warp < kProducerWarps) {
    // Producer warps. Tiles come in batches: first dealt round-robin (tile b + i * grid of
    // the first static_tiles), then, for the tail, claimed from a counter shared by the
    // CTAs, so that SMs that run faster take more of the last tiles. A claim takes kClaim
    // tiles or, guided, about half of this CTA's fair share of the tail still unclaimed
    // (kClaim to 32 tiles): fewer claims, each covering the memory round trips of the
    // next one. Warp 0 resolves a batch (lane i: tile i, from its record; one memory round
    // trip per batch) into the table and publishes its size; then each warp issues the
    // batch's tiles of its parity (k % 2), tile by tile: lane 0 waits for the stage to be
    // free, records the tile's entry and the bytes to expect, and lanes j < nsrc each issue
    // source j's bulk copy. A warp's bulk copies enter the copy engine one stage's worth at
    // a time, so two issuing warps keep twice the copies moving. The two warps meet at a
    // named barrier after each publication and after each batch's issue.
    uint32_t k0 = 0;  // tiles of the CTA issued before the current batch
    bool stop = false, dyn = a.static_tiles == 0;
    uint64_t t0 = blockIdx.x;
    uint32_t cnext = 0, nnext = 0;  // warp 0, lane 0: the claim for the batch after this one
    bool cnext_valid = false;
    const uint64_t tail_tiles = total - a.static_tiles;
    auto claim_size = [&](uint64_t claimed) -> uint32_t {
      if (a.dyn_tail != 2u) return kClaim;
      const uint64_t left = claimed < tail_tiles ? tail_tiles - claimed : 0u;
      const uint64_t q = left / (2ull * gridDim.x);
      return q < kClaim ? kClaim : (q > 32u ? 32u : (uint32_t)q);
    };
    // The tiles of the next batch (lane i: one tile), one batch ahead of their issue, so
    // that the claim's and the records' memory round trips overlap the current batch.
    auto next_batch = [&](uint64_t &t, bool &have) {
      have = false;
      if (!dyn) {
        t = t0 + (uint64_t)lane * gridDim.x;
        have = t < a.static_tiles;
        t0 += 32ull * gridDim.x;
        if (!__any_sync(FULLW, have)) dyn = true;
      }
      if (dyn) {
        uint32_t c = 0, n = 0;
        if (lane == 0) {
          if (cnext_valid) {
            c = cnext;
            n = nnext;
          } else {
            n = claim_size(0);
            c = atomicAdd(&a.st->tail_claim, n);
          }
          nnext = claim_size((uint64_t)c + n);
          cnext = atomicAdd(&a.st->tail_claim, nnext);  // (its value is used next time)
          cnext_valid = true;
        }
        c = __shfl_sync(FULLW, c, 0);
        n = __shfl_sync(FULLW, n, 0);
        t = a.static_tiles + c + lane;
        have = lane < n && t < total;
      }
    };
    auto load_record = [&](uint64_t t, bool have, uint4 w[9]) {
      if (have) {
        const uint32_t e = (uint32_t)(t / a.ntiles);
        const uint4 *rec = reinterpret_cast<const uint4 *>(a.btiles + (t - (uint64_t)e * a.ntiles));
#pragma unroll
        for (uint32_t q = 0; q < 9; ++q) w[q] = ld_nc_v4(rec + q);
      }
    };
    uint64_t tA = 0, tB = 0;
    bool haveA = false, haveB = false;
    uint4 wA[9], wB[9];  // warp 0: the 144-byte records
    bool waited = false;  // the previous kernel in the stream has completed
    auto dep_wait = [&]() {
      if (!waited) griddep_wait();
      waited = true;
    };
    if (warp == 0) {
      if (dyn) dep_wait();  // (a claimed first batch reads the plan's counter)
      next_batch(tA, haveA);
      load_record(tA, haveA, wA);
    }
    for (;;) {
      if (warp == 0) {
        const uint32_t nhave = __popc(__ballot_sync(FULLW, haveA));
        // (one lane reads the abort word, so that the warp takes one decision)
        const bool halt = __shfl_sync(FULLW, (stop || s_abort) ? 1u : 0u, 0) != 0u;
        const uint32_t batch = halt ? 0u : nhave;
        if (haveA && batch) {
          const uint32_t e = (uint32_t)(tA / a.ntiles);
          const uint64_t start = ((uint64_t)wA[0].y << 32) | wA[0].x;
          TileRec &tr = table[(k0 + lane) % kTable];
          tr.nbytes = wA[0].z;
          tr.nsrc = wA[0].w & 0xFFFFu;
          tr.ndst = wA[0].w >> 16;
          const int64_t ioff = (int64_t)(e % (uint32_t)a.in_pool) * a.in_stride + (int64_t)start;
          const int64_t ooff = (int64_t)e * a.out_stride + (int64_t)start;
          constexpr uint64_t kOffMask = (1ull << 56) - 1u;
          // references 0..7 are sources, 8..15 destinations; word q + 1 holds 2q and 2q + 1
#pragma unroll
          for (uint32_t q = 0; q < 8; ++q) {
            const uint64_t ra = ((uint64_t)wA[q + 1].y << 32) | wA[q + 1].x;
            const uint64_t rb = ((uint64_t)wA[q + 1].w << 32) | wA[q + 1].z;
#pragma unroll
            for (uint32_t h2 = 0; h2 < 2; ++h2) {
              const uint64_t r = h2 ? rb : ra;
              const uint32_t i = 2 * q + h2;
              if (i < COLL_BULK_MAX_SRC) {
                tr.src[i] = i < tr.nsrc ? a.ptr.in[(uint32_t)(r >> 56)] + (r & kOffMask) + ioff
                                        : nullptr;
              } else {
                const uint32_t d = i - COLL_BULK_MAX_SRC;
                tr.dst[d] = d < tr.ndst ? a.ptr.out[(uint32_t)(r >> 56)] + (r & kOffMask) + ooff
                                        : nullptr;
              }
            }
          }
        }
        __syncwarp();  // the batch's table entries are written before it is published
        if (batch) dep_wait();  // before the plan's counters and the caller's buffers are touched
        if (lane == 0) s_batch = batch;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kProducerWarps) : "memory");  // published
      const uint32_t batch = s_batch;
      if (batch == 0) break;
      if (warp == 0) {
        next_batch(tB, haveB);
        load_record(tB, haveB, wB);
      } else {
        dep_wait();  // (already satisfied: warp 0 waited before publishing)
      }
      for (uint32_t k = k0 + ((k0 & 1u) != warp ? 1u : 0u); k < k0 + batch && !stop; k += 2) {
        const uint32_t s = k % S, lap = k / S;
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&empty[s], (lap & 1u) ^ 1u, a.spin_ns, &s_abort);
        ok = __shfl_sync(FULLW, ok, 0);
        if (!ok) {
          if (lane == 0) {
            bulk_timeout(a.st, k);
            s_abort = 1;
          }
          stop = true;
          break;
        }
        const uint32_t ent = k % kTable;
        const TileRec &tr = table[ent];
        const uint32_t nb = tr.nbytes, ns = tr.nsrc;
        if (lane == 0) {
          stile[s] = ent;
          mbar_expect_tx(&full[s], ns * nb);
          s_issued[warp] = k + 1;
        }
        __syncwarp();  // the bytes are expected before any copy can complete them
        if (lane < ns)
          bulk_load(data + (size_t)s * stage_bytes + (size_t)lane * a.slot_bytes, tr.src[lane], nb,
                    &full[s]);
      }
      k0 += batch;
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kProducerWarps) : "memory");  // batch issued
      if (warp == 0) {
        tA = tB;
        haveA = haveB;
#pragma unroll
        for (uint32_t q = 0; q < 9; ++q) wA[q] = wB[q];
      }
    }
    // The end: tile k0 does not exist. Once its stage is free, record k0 and complete the
    // stage's barrier with a plain arrival (no bytes), so that the consumers waiting for
    // tile k0 wake, read the count and stop.
    if (warp == 0) {
      dep_wait();  // (a CTA without tiles still updates the plan's counters at the end)
      if (lane == 0) {
        griddep_launch();  // every copy of this CTA is issued: the next kernel may start
        const uint32_t s = k0 % S, lap = k0 / S;
        bool ok = !stop && !s_abort;
        if (ok) ok = mbar_wait(&empty[s], (lap & 1u) ^ 1u, a.spin_ns, &s_abort);
        s_final = k0;
        if (ok) mbar_arrive(&full[s]);
      }
    }
  } else {
    const uint32_t ctid = threadIdx.x - 32 * kProducerWarps;  // consumer thread index
    const uint32_t slot_vec = a.slot_bytes >> 4;
    uint32_t k = 0, s = 0, lap = 0;
    for (;; ++k) {
      const bool ok = __all_sync(FULLW, mbar_wait(&full[s], lap & 1u, a.spin_ns, &s_abort));
      if (ok && k >= s_final) break;  // the producer's end marker, not a tile
      if (!ok) {
        if (lane == 0) bulk_timeout(a.st, k);
        s_abort = 1;
        break;
      }
      const TileRec &h = table[stile[s]];
      const uint32_t nvec = h.nbytes >> 4, nsrc = h.nsrc, ndst = h.ndst;
      const uint4 *sd = reinterpret_cast<const uint4 *>(data + (size_t)s * stage_bytes);
      for (uint32_t v = ctid; v < nvec; v += 32 * kConsumerWarps) {
        uint4 r;
        if constexpr (KIND == 0) {
          r = sd[v];
        } else {
          uint4 x[COLL_BULK_MAX_SRC];
#pragma unroll
          for (uint32_t j = 0; j < COLL_BULK_MAX_SRC; ++j)
            if (j < nsrc) x[j] = sd[(size_t)j * slot_vec + v];
          Vec16Acc<KIND - 1> acc;
          if constexpr (TREE) {
            tree8<KIND - 1>(acc, true, x, nsrc);
          } else {
            acc.init(x[0]);
#pragma unroll
            for (uint32_t j = 1; j < COLL_BULK_MAX_SRC; ++j)
              if (j < nsrc) acc.add(x[j]);
          }
          r = acc.pack();
        }
        for (uint32_t d = 0; d < ndst; ++d) st_cs_v4(h.dst[d] + (size_t)v * 16, r);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      consumed = k + 1;
      if (++s == S) {
        s = 0;
        ++lap;
      }
    }
  }
  __syncthreads();
  if (s_abort && threadIdx.x == 32 * kProducerWarps) {
    // bulk copies issued but not consumed may still be landing in this CTA's shared
    // memory: wait for them (bounded) before the CTA exits. Warp p issued the tiles
    // k = p (mod 2) below s_issued[p].
    const volatile uint32_t never = 0;
    const uint32_t hi = s_issued[0] > s_issued[1] ? s_issued[0] : s_issued[1];
    for (uint32_t k = consumed; k < hi; ++k)
      if (k < s_issued[k & 1u]) mbar_wait(&full[k % S], (k / S) & 1u, 100000000ull, &never);
  }
  if (threadIdx.x == 0) {
    // the last CTA to finish zeroes the tail counters for the plan's next run
    __threadfence();
    if (atomicAdd(&a.st->tail_done, 1u) == gridDim.x - 1u) {
      atomicExch(&a.st->tail_claim, 0u);
      atomicExch(&a.st->tail_done, 0u);
      __threadfence();
    }
  }
}

}  // namespace

uint32_t bulk_smem_bytes(uint32_t stages, uint32_t maxsrc, uint32_t slot_bytes) {
  const uint32_t head = ((16u * stages + 4u * stages) + 127u) & ~127u;
  return head + stages * maxsrc * slot_bytes;
}

cudaError_t launch_bulk(int op, int dtype, const ZcArgs &a, int ctas, cudaStream_t s) {
  const uint64_t total = (uint64_t)a.ntiles * a.n_epochs;
  if (total == 0) return cudaSuccess;
  const int grid = (int)((uint64_t)ctas < total ? (uint64_t)ctas : total);
  const uint32_t smem = bulk_smem_bytes(a.stages, a.maxsrc, a.slot_bytes);
  // Whole rounds of four fifths of the tiles are dealt round-robin and the rest claimed,
  // two at a time (dyn_tail 1) or in guided sizes (dyn_tail 2), else every tile is dealt
  // round-robin. A guided tail pays for its claims only in long enough runs: with fewer than
  // 16 tiles per CTA every tile is dealt.
  ZcArgs la = a;
  const bool tail = a.dyn_tail == 1u || (a.dyn_tail == 2u && total >= 16ull * (uint64_t)grid);
  la.static_tiles = tail ? total * 4 / 5 / (uint64_t)grid * (uint64_t)grid : total;
  if (total - la.static_tiles >= (1ull << 31)) la.static_tiles = total;  // (claim counter)
  const void *fn;
  if (op == COLL_OP_COPY) fn = (const void *)bulk_kernel<0, false>;
  else if (dtype == COLL_BF16) fn = a.tree ? (const void *)bulk_kernel<1, true> : (const void *)bulk_kernel<1, false>;
  else fn = a.tree ? (const void *)bulk_kernel<2, true> : (const void *)bulk_kernel<2, false>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  void *args[] = {(void *)&la};
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace coll
