// All-reduce that allocates nothing: a variant of the staged engine (dual buffers, release /
// acquire epoch flags, fixed rank-order binary32 sum) whose exchange buffers and flags live
// in one fixed file-scope device array instead of memory a plan allocates.
//
// Some callers cannot allocate device memory at the point where they need the collective:
// a serving process that reserved nearly all HBM up front for weights and the KV cache (a
// late cudaMalloc then fails, or fragments that reservation), and latency-critical loops
// where a cudaMalloc/cudaFree pair would add an implicit device synchronisation. This entry
// point serves them; everything it needs beyond the caller's inputs and outputs is in
// g_static_scratch.
//
// g_static_scratch is kStaticScratchBytes on every device that loads the library and stays
// allocated until the process exits. Host code must not pass its name to a kernel (in host
// code the symbol is only a host-side stand-in); the device address is looked up once per
// device with cudaGetSymbolAddress, on the first call made while that device is current
// (make that first call before any stream capture). All calls share the array and it keeps
// the last call's contents: each call clears the flag words it uses before its kernel
// runs, on the caller's stream. Calls that can overlap on the GPU (different streams, or
// no ordering between them) race on the array.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "atom.cuh"
#include "coll_internal.h"

namespace coll {
namespace {

constexpr size_t kStaticScratchBytes = 4u << 20;  // per device
constexpr uint32_t kUnit = 512;                   // bytes per warp piece
constexpr int kMaxDevices = 64;
constexpr unsigned FULLM = 0xFFFFFFFFu;

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
unsigned char *g_scratch_dev[kMaxDevices];  // device address per device, once looked up

struct StaticArgs {
  const char *in[COLL_MAX_RANKS];
  char *out[COLL_MAX_RANKS];
  unsigned long long *flags;  // [2][units][R] epoch words
  uint32_t *abort_word;
  char *xbuf;                 // [2][units][R][kUnit]
  int32_t *status;            // caller's status word or null
  uint32_t R, units, last_bytes;
  int32_t n_epochs, in_pool;
  int64_t in_stride, out_stride;
  uint64_t spin_ns;
};

__device__ __forceinline__ bool wait_epoch(const unsigned long long *f, uint32_t E,
                                           const uint32_t *abort_word, uint64_t limit) {
  uint64_t t0 = 0;
  for (uint32_t k = 0;; ++k) {
    if ((uint32_t)ld_acquire_u64(f) == E) return true;
    if ((k & 31u) == 31u) {
      const uint64_t now = globaltimer();
      if (t0 == 0) t0 = now;
      else if (now - t0 > limit) return false;
      if (ld_relaxed_u32(abort_word)) return false;
    }
  }
}

// DT: 0 bf16, 1 f32. One warp per (rank r, piece k): stage piece k of rank r's input into
// its exchange slot, notify, wait for every rank's slot of piece k, reduce in rank order.
template <int DT>
__global__ void __launch_bounds__(32) static_allreduce_kernel(const StaticArgs a) {
  const uint32_t w = blockIdx.x;
  const uint32_t r = w / a.units, k = w % a.units;
  if (r >= a.R) return;
  const uint32_t lane = threadIdx.x;
  const uint32_t nb = (k + 1 == a.units) ? a.last_bytes : kUnit;
  const bool active = lane < (nb >> 4);
  for (int i = 0; i < a.n_epochs; ++i) {
    const uint32_t E = (uint32_t)i + 1u;
    const uint32_t b = E & 1u;
    const size_t row = ((size_t)b * a.units + k) * a.R;  // flags/slots of piece k, parity b
    if (active) {
      const uint4 x = ld_nc_v4(a.in[r] + (int64_t)(i % a.in_pool) * a.in_stride +
                               (size_t)k * kUnit + lane * 16);
      st_v4(a.xbuf + (row + r) * kUnit + lane * 16, x);
    }
    __syncwarp();
    if (lane == 0) st_release_u64(a.flags + row + r, E);
    bool ok = true;
    for (uint32_t j = lane; j < a.R; j += 32)
      ok = ok && wait_epoch(a.flags + row + j, E, a.abort_word, a.spin_ns);
    if (!__all_sync(FULLM, ok)) {
      if (lane == 0) {
        if (a.status) atomicCAS(a.status, 0, COLL_ETIMEDOUT);
        st_relaxed_u32(a.abort_word, 1u);
      }
      return;
    }
    // lane j's acquire of rank j's flag must order every lane's loads of rank j's slot: a
    // vote orders nothing in memory, the warp barrier does
    __syncwarp();
    Vec16Acc<DT> acc;
    for (uint32_t j0 = 0; j0 < a.R; j0 += 8) {
      uint4 x[8];
      const uint32_t jn = a.R - j0 < 8 ? a.R - j0 : 8;
#pragma unroll
      for (uint32_t j = 0; j < 8; ++j)
        if (j < jn && active) x[j] = ld_relaxed_v4(a.xbuf + (row + j0 + j) * kUnit + lane * 16);
      if (active) {
#pragma unroll
        for (uint32_t j = 0; j < 8; ++j)
          if (j < jn) {
            if (j0 + j == 0) acc.init(x[j]); else acc.add(x[j]);
          }
      }
    }
    if (active)
      st_v4(a.out[r] + (int64_t)i * a.out_stride + (size_t)k * kUnit + lane * 16, acc.pack());
  }
}

int scratch_for_current_device(unsigned char **p) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return COLL_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return COLL_EINVAL;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_dev[dev]) {
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_static_scratch) != cudaSuccess || !addr) {
      cudaGetLastError();
      return COLL_ECUDA;
    }
    g_scratch_dev[dev] = static_cast<unsigned char *>(addr);
  }
  *p = g_scratch_dev[dev];
  return COLL_OK;
}

}  // namespace
}  // namespace coll

extern "C" int coll_allreduce_static(int R, int dtype, void *const *in, void *const *out,
                                     uint64_t count, int n_epochs, int64_t in_epoch_stride,
                                     int in_pool, int64_t out_epoch_stride, int32_t *status,
                                     void *stream) {
  using namespace coll;
  if (R < 1 || R > COLL_MAX_RANKS || (dtype != COLL_BF16 && dtype != COLL_F32) || !in || !out ||
      count == 0 || n_epochs < 1 || in_pool < 1)
    return COLL_EINVAL;
  const uint64_t es = dtype == COLL_BF16 ? 2 : 4;
  if (count > kStaticScratchBytes / es) return COLL_ETOOBIG;  // (and count * es cannot wrap)
  const uint64_t bytes = count * es;
  if (bytes & 15u) return COLL_EALIGN;
  if ((uint64_t)(in_epoch_stride < 0 ? -in_epoch_stride : in_epoch_stride) & 15u ||
      (uint64_t)(out_epoch_stride < 0 ? -out_epoch_stride : out_epoch_stride) & 15u)
    return COLL_EALIGN;
  for (int r = 0; r < R; ++r) {
    if (!in[r] || !out[r]) return COLL_EINVAL;
    if (((uintptr_t)in[r] & 15u) || ((uintptr_t)out[r] & 15u)) return COLL_EALIGN;
  }
  const uint64_t units = (bytes + kUnit - 1) / kUnit;
  const uint64_t flag_bytes = (2 * units * R * 8 + 255) & ~255ull;
  const uint64_t need = flag_bytes + 256 + 2 * units * R * kUnit;
  if (need > kStaticScratchBytes) return COLL_ETOOBIG;
  const uint64_t warps = units * R;
  int dev = 0, sms = 0, per_sm = 0;
  const void *fn = dtype == COLL_BF16 ? (const void *)static_allreduce_kernel<0>
                                      : (const void *)static_allreduce_kernel<1>;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, 32, 0) != cudaSuccess)
    return COLL_ECUDA;
  if (warps > (uint64_t)per_sm * sms) return COLL_ETOOBIG;  // every warp must be co-resident
  unsigned char *base = nullptr;
  if (int e = scratch_for_current_device(&base)) return e;
  StaticArgs a;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < R; ++r) {
    a.in[r] = static_cast<const char *>(in[r]);
    a.out[r] = static_cast<char *>(out[r]);
  }
  a.flags = reinterpret_cast<unsigned long long *>(base);
  a.abort_word = reinterpret_cast<uint32_t *>(base + flag_bytes);
  a.xbuf = reinterpret_cast<char *>(base + flag_bytes + 256);
  a.status = status;
  a.R = (uint32_t)R;
  a.units = (uint32_t)units;
  a.last_bytes = (uint32_t)(bytes - (units - 1) * kUnit);
  a.n_epochs = n_epochs;
  a.in_pool = in_pool;
  a.in_stride = in_epoch_stride;
  a.out_stride = out_epoch_stride;
  a.spin_ns = 2000000000ull;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the flags and the abort word must start at zero; the status word too
  if (cudaMemsetAsync(base, 0, flag_bytes + 256, s) != cudaSuccess ||
      (status && cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess)) {
    cudaGetLastError();
    return COLL_ECUDA;
  }
  void *args[] = {(void *)&a};
  if (cudaLaunchCooperativeKernel(fn, dim3((unsigned)warps), dim3(32), args, 0, s) !=
      cudaSuccess) {
    cudaGetLastError();
    return COLL_ECUDA;
  }
  return COLL_OK;
}
