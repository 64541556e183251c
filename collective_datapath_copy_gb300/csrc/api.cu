// C ABI: plan lifecycle and runs (see include/coll.h for the contract of each call).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <memory>
#include <new>
#include <vector>

#include "coll_internal.h"
#include "engine.cuh"

struct coll_plan_s {
  coll_compiled c;
  int device = 0;
  int num_sms = 0;
  char *d_tables = nullptr;  // one allocation for every read-only table
  coll_ref_t *d_refs = nullptr;
  coll_job_t *d_jobs = nullptr;
  coll_tile_t *d_tiles = nullptr;
  coll_btile_t *d_btiles = nullptr;
  coll_unit_t *d_units = nullptr;
  coll_item_t *d_sitems = nullptr, *d_citems = nullptr, *d_pitems = nullptr;
  coll_warp_t *d_warps = nullptr;
  char *d_xbuf = nullptr;
  unsigned long long *d_pflag = nullptr;
  uint32_t *d_cflag = nullptr;
  char *d_rbuf = nullptr;      // two-shot pull: reduced pieces [parity][unit]
  uint32_t *d_rflag = nullptr; // two-shot pull: [parity][unit] epoch of the reduced piece
  uint32_t *d_dflag = nullptr; // two-shot pull: [n_dflag] epoch each consumer has pulled
  coll_dev_status_t *d_status = nullptr;
  uint64_t *d_stamps = nullptr;
  uint32_t *d_dbg = nullptr;
  uint32_t *d_rank_done = nullptr;
  uint32_t stamp_cap = 0;
  uint64_t epochs_issued = 0;
  cudaEvent_t done = nullptr;
  bool ran = false;
  bool captured = false;  // a run was captured into a graph: status waits for the device
  int last_epochs = 0;
  int gemv_cap = -1;  // co-resident fused-producer CTAs; queried on the first fused run
  bool single_items = false;  // every warp has one stage and one consume item
  // tensor maps of the last fused run's weight matrices, and what they were encoded for
  std::unique_ptr<coll::GemvMaps> gmaps;
  std::vector<const void *> gmaps_wt;
  uint32_t gmaps_k = 0;
};

namespace {

template <typename T>
size_t table_bytes(const std::vector<T> &v) {
  return (v.size() * sizeof(T) + 255) & ~(size_t)255;
}

template <typename T>
T *carve(char *base, size_t &off, const std::vector<T> &v) {
  T *p = reinterpret_cast<T *>(base + off);
  off += table_bytes(v);
  return v.empty() ? nullptr : p;
}

void release(coll_plan_s *p) {
  if (!p) return;
  if (p->done) {
    cudaEventSynchronize(p->done);
    cudaEventDestroy(p->done);
  }
  cudaFree(p->d_tables);
  cudaFree(p->d_xbuf);
  cudaFree(p->d_pflag);
  cudaFree(p->d_cflag);
  cudaFree(p->d_rbuf);
  cudaFree(p->d_rflag);
  cudaFree(p->d_dflag);
  cudaFree(p->d_status);
  cudaFree(p->d_stamps);
  cudaFree(p->d_dbg);
  cudaFree(p->d_rank_done);
  delete p;
}

int zero_state(coll_plan_s *p) {
  const coll_compiled &c = p->c;
  if (p->d_pflag && cudaMemset(p->d_pflag, 0, (size_t)c.n_pflag * 2 * 8) != cudaSuccess)
    return COLL_ECUDA;
  if (p->d_cflag && cudaMemset(p->d_cflag, 0, (size_t)c.n_cflag * 4) != cudaSuccess)
    return COLL_ECUDA;
  if (p->d_dbg && cudaMemset(p->d_dbg, 0, (size_t)c.units.size() * 4) != cudaSuccess)
    return COLL_ECUDA;
  if (p->d_rflag && cudaMemset(p->d_rflag, 0, c.units.size() * 2 * 4) != cudaSuccess)
    return COLL_ECUDA;
  if (p->d_dflag && cudaMemset(p->d_dflag, 0, (size_t)c.n_dflag * 4) != cudaSuccess)
    return COLL_ECUDA;
  if (p->d_rank_done && cudaMemset(p->d_rank_done, 0, (size_t)c.R * 4) != cudaSuccess)
    return COLL_ECUDA;
  // tagged data keeps its epochs in the exchange words: epochs restart at 1 after a reset
  if (c.cfg.protocol == COLL_PROTO_LL && p->d_xbuf &&
      cudaMemset(p->d_xbuf, 0, (size_t)c.xpar_bytes * 2) != cudaSuccess)
    return COLL_ECUDA;
  if (cudaMemset(p->d_status, 0, sizeof(coll_dev_status_t)) != cudaSuccess) return COLL_ECUDA;
  p->epochs_issued = 0;
  return COLL_OK;
}

bool overlaps(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) {
  return a0 < b1 && b0 < a1;
}

// The CUDA driver API's tensor-map encoder, looked up once through the runtime (no link to the
// driver library).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      p = nullptr;
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// Tensor maps of the fused run's weight matrices W_r ([k rows][in_len[r] bf16], rows
// in_bytes[r] apart), boxes of one unit's columns (at most 256) x 64 rows; reused while the
// run's matrices and k stay the same.
// Bytes per staged weight row of the fused producer: the plan's unit.
uint32_t gemv_pitch(const coll_compiled &c) {
  return c.cfg.unit_bytes ? (uint32_t)c.cfg.unit_bytes : 512u;
}

int gemv_maps(coll_plan_s *p, const void *const *wt, uint32_t k) {
  const coll_compiled &c = p->c;
  std::vector<const void *> key(wt, wt + c.R);
  if (p->gmaps && p->gmaps_k == k && p->gmaps_wt == key) return COLL_OK;
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return COLL_ECUDA;
  if (!p->gmaps) {
    p->gmaps.reset(new (std::nothrow) coll::GemvMaps());
    if (!p->gmaps) return COLL_ENOMEM;
  }
  memset(p->gmaps.get(), 0, sizeof(coll::GemvMaps));
  p->gmaps_wt.clear();
  for (int r = 0; r < c.R; ++r) {
    if (!c.in_used[r]) continue;
    const cuuint64_t dims[2] = {(cuuint64_t)(c.in_bytes[r] / 2), (cuuint64_t)k};
    const cuuint64_t strides[1] = {(cuuint64_t)c.in_bytes[r]};
    const cuuint32_t box[2] = {gemv_pitch(c) / 2u, 64};
    const cuuint32_t estr[2] = {1, 1};
    if (dims[0] > 0xFFFFFFFFull || strides[0] >= (1ull << 40)) return COLL_EINVAL;
    if (encode(&p->gmaps->m[r], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(wt[r]),
               dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return COLL_EINVAL;
  }
  p->gmaps_wt = key;
  p->gmaps_k = k;
  return COLL_OK;
}

}  // namespace

extern "C" int coll_plan(coll_plan_t *out, int R, int op, int dtype, const coll_seg_t *in_segs,
                         size_t n_in, const uint64_t *in_len, const coll_seg_t *out_segs,
                         size_t n_out, const uint64_t *out_len, const coll_config_t *cfg) {
  if (!out) return COLL_EINVAL;
  *out = nullptr;
  coll_plan_s *p = new (std::nothrow) coll_plan_s();
  if (!p) return COLL_ENOMEM;
  if (cudaGetDevice(&p->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) {
    delete p;
    return COLL_ECUDA;
  }
  int max_ctas = coll_default_max_warps();
  const int eop = (op == COLL_OP_SUM) ? COLL_OP_SUM : COLL_OP_COPY;
  const int eproto = cfg ? cfg->protocol : COLL_PROTO_SPEC;
  const int edp = cfg ? cfg->datapath : COLL_DP_ONESHOT;
  if (coll::engine_max_coresident(eop, dtype == COLL_F32 ? COLL_F32 : COLL_BF16, eproto, edp,
                                  &max_ctas) !=
      cudaSuccess) {
    delete p;
    return COLL_ECUDA;
  }
  int e = coll_compile(R, op, dtype, in_segs, n_in, in_len, out_segs, n_out, out_len, cfg,
                       max_ctas, p->num_sms, &p->c);
  if (e) {
    delete p;
    return e;
  }
  coll_compiled &c = p->c;
  if (!c.cfg.zero_copy && c.warps.size() > (size_t)max_ctas) {  // must all be co-resident
    delete p;
    return COLL_EINVAL;
  }
  const size_t tb = table_bytes(c.refs) + table_bytes(c.jobs) + table_bytes(c.tiles) +
                    table_bytes(c.btiles) +
                    table_bytes(c.units) + table_bytes(c.sitems) + table_bytes(c.citems) +
                    table_bytes(c.pitems) + table_bytes(c.warps);
  std::vector<char> host(tb ? tb : 256, 0);
  size_t off = 0;
  auto put = [&](const auto &v) {
    if (!v.empty()) memcpy(host.data() + off, v.data(), v.size() * sizeof(v[0]));
    off += table_bytes(v);
  };
  put(c.refs); put(c.jobs); put(c.tiles); put(c.btiles); put(c.units); put(c.sitems);
  put(c.citems);
  put(c.pitems); put(c.warps);
  bool ok = cudaMalloc(&p->d_tables, host.size()) == cudaSuccess &&
            cudaMemcpy(p->d_tables, host.data(), host.size(), cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMalloc(&p->d_status, sizeof(coll_dev_status_t)) == cudaSuccess &&
            cudaEventCreateWithFlags(&p->done, cudaEventDisableTiming) == cudaSuccess;
  if (ok) {
    off = 0;
    p->d_refs = carve(p->d_tables, off, c.refs);
    p->d_jobs = carve(p->d_tables, off, c.jobs);
    p->d_tiles = carve(p->d_tables, off, c.tiles);
    p->d_btiles = carve(p->d_tables, off, c.btiles);
    p->d_units = carve(p->d_tables, off, c.units);
    p->d_sitems = carve(p->d_tables, off, c.sitems);
    p->d_citems = carve(p->d_tables, off, c.citems);
    p->d_pitems = carve(p->d_tables, off, c.pitems);
    p->d_warps = carve(p->d_tables, off, c.warps);
  }
  if (ok && !c.cfg.zero_copy) {
    const bool dual = c.cfg.protocol != COLL_PROTO_BARRIER;
    const size_t xb = (size_t)c.xpar_bytes * (dual ? 2 : 1);
    ok = (xb == 0 || cudaMalloc(&p->d_xbuf, xb) == cudaSuccess) &&
         (c.n_pflag == 0 || cudaMalloc(&p->d_pflag, (size_t)c.n_pflag * 2 * 8) == cudaSuccess) &&
         (c.n_cflag == 0 || cudaMalloc(&p->d_cflag, (size_t)c.n_cflag * 4) == cudaSuccess);
    if (ok && xb) ok = cudaMemset(p->d_xbuf, 0, xb) == cudaSuccess;
    if (ok && c.rpar_bytes)
      ok = cudaMalloc(&p->d_rbuf, (size_t)c.rpar_bytes * (dual ? 2 : 1)) == cudaSuccess &&
           cudaMalloc(&p->d_rflag, c.units.size() * 2 * 4) == cudaSuccess &&
           cudaMalloc(&p->d_dflag, (size_t)c.n_dflag * 4) == cudaSuccess;
    if (ok && c.cfg.chain) ok = cudaMalloc(&p->d_rank_done, (size_t)c.R * 4) == cudaSuccess;
    if (ok && (c.cfg.inject_flags & COLL_INJECT_SPEC_PAUSE) && !c.units.empty())
      ok = cudaMalloc(&p->d_dbg, c.units.size() * 4) == cudaSuccess;
    if (ok && c.cfg.record_stamps && c.cfg.stamp_capacity) {
      p->stamp_cap = c.cfg.stamp_capacity;
      const size_t per = c.cfg.record_stamps == 2 ? 4 : 1;
      ok = cudaMalloc(&p->d_stamps, ((size_t)p->stamp_cap * per + 1) * 8) == cudaSuccess;
    }
  }
  if (ok) ok = zero_state(p) == COLL_OK;
  p->single_items = !c.warps.empty();
  for (const coll_warp_t &w : c.warps)
    if (w.s1 - w.s0 != 1 || w.c1 - w.c0 != 1) p->single_items = false;
  if (!ok) {
    cudaGetLastError();
    release(p);
    return COLL_ECUDA;
  }
  if (cudaDeviceSynchronize() != cudaSuccess) {
    release(p);
    return COLL_ECUDA;
  }
  *out = p;
  return COLL_OK;
}

extern "C" int coll_plan_info(coll_plan_t p, coll_plan_info_t *info) {
  if (!p || !info) return COLL_EINVAL;
  coll_fill_info(p->c, info);
  return COLL_OK;
}

// One run. With wt != null (fused producer) `in` holds the GEMV vectors x_r of k elements
// and the stage computes each payload piece as W_r x_r instead of loading it.
static int run_impl(coll_plan_s *p, void *const *in, void *const *out, int n_epochs,
                    int64_t in_epoch_stride, int in_pool, int64_t out_epoch_stride,
                    void *stream, const void *const *wt, uint32_t k) {
  if (!p || !in || !out || n_epochs < 1 || in_pool < 1) return COLL_EINVAL;
  const coll_compiled &c = p->c;
  const int R = c.R;
  if (wt) {
    // the compute takes the rows sixteen at a time and x is staged whole: k is a multiple
    // of 16, at most 8192
    if (c.cfg.zero_copy || c.dtype != COLL_BF16 || k < 16 || (k & 15u) || k > 8192)
      return COLL_EINVAL;
    if (c.cfg.protocol == COLL_PROTO_LL) return COLL_EINVAL;  // tagged data is not fused
    for (int r = 0; r < R; ++r) {
      if (!c.in_used[r]) continue;
      if (!wt[r]) return COLL_EINVAL;
      if (((uintptr_t)wt[r] & 15u) || (c.in_bytes[r] & 15u)) return COLL_EALIGN;
    }
    // the fused CTAs are larger (eight warps and a shared-memory ring): all must still fit
    if (p->gemv_cap < 0 &&
        coll::engine_gemv_max_coresident(c.rpar_bytes != 0, &p->gemv_cap) != cudaSuccess) {
      cudaGetLastError();
      p->gemv_cap = -1;
      return COLL_ECUDA;
    }
    if (c.warps.size() > (size_t)p->gemv_cap) return COLL_EINVAL;
    if (const int e = gemv_maps(p, wt, k)) return e;
  }
  // bytes of one rank's per-epoch input as the kernel reads it
  auto in_span = [&](int r) -> uint64_t { return wt ? (uint64_t)k * 2 : c.in_bytes[r]; };
  coll::RankPtrs ptr;
  memset(&ptr, 0, sizeof(ptr));
  // spans touched over all epochs, for the aliasing check
  std::vector<uintptr_t> i0(R, 0), i1(R, 0), o0(R, 0), o1(R, 0);
  const bool staged = !c.cfg.zero_copy;
  for (int r = 0; r < R; ++r) {
    if (c.in_used[r]) {
      if (!in[r]) return COLL_EINVAL;
      if (staged && ((uintptr_t)in[r] & 15u)) return COLL_EALIGN;
      const int64_t lo = std::min<int64_t>(0, in_epoch_stride * (in_pool - 1));
      const int64_t hi = std::max<int64_t>(0, in_epoch_stride * (in_pool - 1));
      i0[r] = (uintptr_t)in[r] + lo;
      i1[r] = (uintptr_t)in[r] + hi + in_span(r);
    }
    if (c.out_used[r]) {
      if (!out[r]) return COLL_EINVAL;
      if (staged && ((uintptr_t)out[r] & 15u)) return COLL_EALIGN;
      const int64_t lo = std::min<int64_t>(0, out_epoch_stride * (n_epochs - 1));
      const int64_t hi = std::max<int64_t>(0, out_epoch_stride * (n_epochs - 1));
      o0[r] = (uintptr_t)out[r] + lo;
      o1[r] = (uintptr_t)out[r] + hi + c.out_bytes[r];
    }
    ptr.in[r] = (const char *)in[r];
    ptr.out[r] = (char *)out[r];
  }
  if (staged && (((uint64_t)(in_epoch_stride < 0 ? -in_epoch_stride : in_epoch_stride) & 15u) ||
                 ((uint64_t)(out_epoch_stride < 0 ? -out_epoch_stride : out_epoch_stride) & 15u)))
    return COLL_EALIGN;
  for (int r = 0; r < R; ++r) {
    if (!c.out_used[r]) continue;
    for (int q = 0; q < R; ++q) {
      if (c.in_used[q] && overlaps(o0[r], o1[r], i0[q], i1[q])) return COLL_EOVERLAP;
      if (wt && c.in_used[q] &&
          overlaps(o0[r], o1[r], (uintptr_t)wt[q], (uintptr_t)wt[q] + (uint64_t)k * c.in_bytes[q]))
        return COLL_EOVERLAP;
      if (q != r && c.out_used[q] && overlaps(o0[r], o1[r], o0[q], o1[q])) return COLL_EOVERLAP;
    }
    // an output buffer reused across epochs must not overlap itself between epochs
    if (out_epoch_stride != 0 && n_epochs > 1 &&
        (uint64_t)(out_epoch_stride < 0 ? -out_epoch_stride : out_epoch_stride) < c.out_bytes[r])
      return COLL_EOVERLAP;
  }
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t err;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return COLL_ECUDA;
  const bool capturing = cs != cudaStreamCaptureStatusNone;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != p->device) return COLL_EINVAL;
  if (c.cfg.zero_copy) {
    coll::ZcArgs a;
    memset(&a, 0, sizeof(a));
    a.ptr = ptr;
    a.jobs = p->d_jobs;
    a.refs = p->d_refs;
    a.tiles = p->d_tiles;
    a.btiles = p->d_btiles;
    a.ntiles = (uint32_t)c.tiles.size();
    a.n_epochs = (uint32_t)n_epochs;
    a.in_pool = in_pool;
    a.in_stride = in_epoch_stride;
    a.out_stride = out_epoch_stride;
    a.st = p->d_status;
    a.spin_ns = c.cfg.spin_limit_ns ? c.cfg.spin_limit_ns : 2000000000ull;
    a.tree = c.cfg.reduce_order == COLL_ORDER_TREE ? 1u : 0u;
    bool bulk = c.bulk;
    if (bulk) {  // the bulk copies need 16-byte-aligned bases and strides at run time
      for (int r = 0; r < R && bulk; ++r) {
        if (c.in_used[r] && ((uintptr_t)in[r] & 15u)) bulk = false;
        if (c.out_used[r] && ((uintptr_t)out[r] & 15u)) bulk = false;
      }
      if (((uint64_t)in_epoch_stride & 15u) || ((uint64_t)out_epoch_stride & 15u)) bulk = false;
    }
    if (bulk) {
      a.slot_bytes = c.bulk_slot;
      a.stages = c.bulk_stages;
      a.maxsrc = c.bulk_maxsrc;
      a.dyn_tail = c.bulk_tail;
      err = coll::launch_bulk(c.op, c.dtype, a, c.cfg.ctas ? c.cfg.ctas : p->num_sms, s);
    } else {
      const int ctas = c.cfg.ctas ? c.cfg.ctas : 3 * p->num_sms;
      const int keep = c.zc_keep ? 1 : 0;
      err = coll::launch_zero_copy(c.op, c.dtype, keep, a, ctas, s);
    }
  } else {
    if (p->epochs_issued + (uint64_t)n_epochs >= 0xFFFFFFF0ull) return COLL_EINVAL;  // reset first
    coll::EngArgs a;
    memset(&a, 0, sizeof(a));
    a.ptr = ptr;
    a.units = p->d_units;
    a.sitems = p->d_sitems;
    a.citems = p->d_citems;
    a.warps = p->d_warps;
    a.refs = p->d_refs;
    a.xbuf = p->d_xbuf;
    a.xpar = c.xpar_bytes;
    a.pflag = p->d_pflag;
    a.cflag = p->d_cflag;
    a.pitems = p->d_pitems;
    a.rbuf = p->d_rbuf;
    a.rpar = c.rpar_bytes;
    a.rflag = p->d_rflag;
    a.dflag = p->d_dflag;
    a.n_units = (uint32_t)c.units.size();
    a.st = p->d_status;
    a.stamps = p->d_stamps;
    a.dbg = p->d_dbg;
    a.rank_done = p->d_rank_done;
    a.chain = c.cfg.chain;
    a.stamp_cap = p->stamp_cap;
    a.stamp_phases = c.cfg.record_stamps == 2 ? 1u : 0u;
    a.n_pflag = c.n_pflag;
    a.nwarps = (uint32_t)c.warps.size();
    a.n_epochs = n_epochs;
    a.in_pool = in_pool;
    // A captured run is replayed with the epochs it was captured with. So once a plan has
    // been captured, every run (the captured one, each of its replays, and later direct
    // runs) first clears the plan's flags on the stream and counts epochs from 1 again:
    // flags left by an earlier replay can then never pass for this run's.
    const bool restart = capturing || p->captured;
    if (restart) {
      const size_t nu = c.units.size();
      if ((p->d_pflag && cudaMemsetAsync(p->d_pflag, 0, (size_t)c.n_pflag * 2 * 8, s)) ||
          (p->d_cflag && cudaMemsetAsync(p->d_cflag, 0, (size_t)c.n_cflag * 4, s)) ||
          (p->d_rflag && cudaMemsetAsync(p->d_rflag, 0, nu * 2 * 4, s)) ||
          (p->d_dflag && cudaMemsetAsync(p->d_dflag, 0, (size_t)c.n_dflag * 4, s)) ||
          (p->d_dbg && cudaMemsetAsync(p->d_dbg, 0, nu * 4, s)) ||
          (p->d_rank_done && cudaMemsetAsync(p->d_rank_done, 0, (size_t)c.R * 4, s)) ||
          // tagged data keeps its epochs in the exchange words themselves
          (c.cfg.protocol == COLL_PROTO_LL && p->d_xbuf &&
           cudaMemsetAsync(p->d_xbuf, 0, (size_t)c.xpar_bytes * 2, s))) {
        cudaGetLastError();
        return COLL_ECUDA;
      }
    }
    a.epoch_base = restart ? 0u : (uint32_t)p->epochs_issued;
    a.in_stride = in_epoch_stride;
    a.out_stride = out_epoch_stride;
    a.protocol = c.cfg.protocol;
    a.spec_check = c.cfg.spec_check;
    a.spec_delay_ns =
        c.cfg.protocol != COLL_PROTO_SPEC ? 0u
        : c.cfg.spec_delay_ns >= 0      ? (uint32_t)c.cfg.spec_delay_ns
        : c.cfg.spec_check == COLL_SPEC_TAGGED_RELAXED ? 200u : 0u;
    // the default window of the fence-free check adapts per warp; a set one stays fixed
    a.spec_adapt = c.cfg.protocol == COLL_PROTO_SPEC && c.cfg.spec_delay_ns < 0 &&
                   c.cfg.spec_check == COLL_SPEC_TAGGED_RELAXED;
    a.spin_ns = c.cfg.spin_limit_ns ? c.cfg.spin_limit_ns : 2000000000ull;
    a.inject_flags = c.cfg.inject_flags;
    a.inject_seed = c.cfg.inject_seed;
    a.inject_rank = c.cfg.inject_rank;
    a.inject_prob_ppm = c.cfg.inject_prob_ppm;
    a.inject_max_ns = c.cfg.inject_max_ns;
    a.inject_start_ns = c.cfg.inject_start_ns;
    a.inject_pause_ns = c.cfg.inject_pause_ns;
    a.R = R;
    a.single_items = p->single_items ? 1u : 0u;
    if (wt) {
      for (int r = 0; r < R; ++r) {
        a.wt[r] = static_cast<const char *>(wt[r]);
        a.wt_stride[r] = (int64_t)c.in_bytes[r];
      }
      a.gemv_k = k;
      a.gemv_pitch = gemv_pitch(c);
      a.gemv_slots = coll::gemv_ring_slots(a.gemv_pitch);
    }
    err = coll::launch_engine(c.op, c.dtype, a, wt ? p->gmaps.get() : nullptr, s);
    if (err == cudaSuccess && !restart) p->epochs_issued += (uint64_t)n_epochs;
  }
  if (err != cudaSuccess) {
    cudaGetLastError();
    return COLL_ECUDA;
  }
  // Inside a stream capture the completion event is not recorded (a captured record
  // cannot be waited on from outside the graph); coll_status then waits for the device.
  if (!capturing) {
    if (cudaEventRecord(p->done, s) != cudaSuccess) return COLL_ECUDA;
    p->ran = true;
  } else {
    p->ran = false;
    p->captured = true;
  }
  p->last_epochs = n_epochs;
  return COLL_OK;
}

extern "C" int coll_run(coll_plan_t p, void *const *in, void *const *out, int n_epochs,
                        int64_t in_epoch_stride, int in_pool, int64_t out_epoch_stride,
                        void *stream) {
  return run_impl(p, in, out, n_epochs, in_epoch_stride, in_pool, out_epoch_stride, stream,
                  nullptr, 0);
}

extern "C" int coll_run_gemv(coll_plan_t p, const void *const *wt, void *const *x, int k,
                             void *const *out, int n_epochs, int64_t x_epoch_stride, int x_pool,
                             int64_t out_epoch_stride, void *stream) {
  if (!wt || k < 1) return COLL_EINVAL;
  return run_impl(p, x, out, n_epochs, x_epoch_stride, x_pool, out_epoch_stride, stream, wt,
                  (uint32_t)k);
}

static int wait_last(coll_plan_s *p) {
  if (p->ran && cudaEventSynchronize(p->done) != cudaSuccess) return COLL_ECUDA;
  if (p->captured && cudaDeviceSynchronize() != cudaSuccess) return COLL_ECUDA;
  return COLL_OK;
}

extern "C" int coll_status(coll_plan_t p, coll_stats_t *st) {
  if (!p) return COLL_EINVAL;
  if (wait_last(p)) return COLL_ECUDA;
  coll_dev_status_t d;
  if (cudaMemcpy(&d, p->d_status, sizeof(d), cudaMemcpyDeviceToHost) != cudaSuccess)
    return COLL_ECUDA;
  if (st) {
    memset(st, 0, sizeof(*st));
    st->status = d.status;
    st->fail_rank = d.status ? d.fail_rank : -1;
    st->fail_unit = d.status ? d.fail_unit : -1;
    st->fail_where = d.fail_where;
    st->fail_epoch = d.fail_epoch;
    st->epochs = d.status ? 0 : p->epochs_issued;
    st->spec_checks = d.spec_checks;
    st->spec_retries = d.spec_retries;
  }
  return d.status;
}

extern "C" int64_t coll_stamps(coll_plan_t p, uint64_t *host, int64_t n) {
  if (!p || !host || n < 0) return COLL_EINVAL;
  if (!p->d_stamps) return 0;
  if (wait_last(p)) return COLL_ECUDA;
  const int64_t per = p->c.cfg.record_stamps == 2 ? 4 : 1;
  int64_t m = std::min<int64_t>(
      n, (int64_t)std::min<uint32_t>(p->stamp_cap, (uint32_t)p->last_epochs) * per + 1);
  if (cudaMemcpy(host, p->d_stamps, (size_t)m * 8, cudaMemcpyDeviceToHost) != cudaSuccess)
    return COLL_ECUDA;
  return m;
}

extern "C" int coll_reset(coll_plan_t p) {
  if (!p) return COLL_EINVAL;
  if (wait_last(p)) return COLL_ECUDA;
  int e = zero_state(p);
  if (e) return e;
  return cudaDeviceSynchronize() == cudaSuccess ? COLL_OK : COLL_ECUDA;
}

extern "C" int coll_free(coll_plan_t p) {
  if (!p) return COLL_OK;
  release(p);
  return COLL_OK;
}

extern "C" const char *coll_strerror(int code) {
  switch (code) {
    case COLL_OK: return "success";
    case COLL_EINVAL: return "invalid argument";
    case COLL_ENAME: return "a consumed name has no producer (or several, for copy)";
    case COLL_ELEN: return "segments with one name have different lengths";
    case COLL_EBOUNDS: return "segment out of its buffer's bounds";
    case COLL_EOVERLAP: return "overlapping output segments or buffers";
    case COLL_EALIGN: return "staged plans need 16-byte-aligned segments, buffers and strides";
    case COLL_ECUDA: return "CUDA runtime error";
    case COLL_ETIMEDOUT: return "a bounded device wait expired";
    case COLL_EDEVICE: return "inconsistent device state";
    case COLL_ENOMEM: return "out of memory";
    case COLL_ETOOBIG: return "request exceeds the fixed static scratch array or co-residency";
    default: return "unknown error";
  }
}

extern "C" int coll_probe_flag_rtt(int peer_block, int iters, uint64_t *ns_total, int *sm_a,
                                   int *sm_b) {
  if (peer_block < 1 || iters < 1 || !ns_total) return COLL_EINVAL;
  unsigned long long *d = nullptr;
  if (cudaMalloc(&d, 1024) != cudaSuccess) return COLL_ECUDA;
  unsigned long long h[8] = {0};
  int rc = COLL_OK;
  if (cudaMemset(d, 0, 1024) != cudaSuccess ||
      coll::launch_probe_rtt(d, (uint32_t)iters, (uint32_t)peer_block, d + 96, 1000000000ull,
                             nullptr) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(h, d + 96, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    rc = COLL_ECUDA;
  }
  cudaFree(d);
  if (rc) return rc;
  if (h[4]) return COLL_ETIMEDOUT;
  *ns_total = h[0];
  if (sm_a) *sm_a = (int)h[2];
  if (sm_b) *sm_b = (int)h[3];
  return COLL_OK;
}
