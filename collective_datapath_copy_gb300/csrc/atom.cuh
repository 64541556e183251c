// Atom: the two datapath primitives of a collective, copy and reduce, for sm_103a.
//
// Source: Purlin article, figure "Purlin separates the collective stack" and section
// "The Purlin PDF describes a three-layer design": under the shared orchestration sits a
// hardware-specific datapath that implements exactly two data movement primitives, copy
// and reduce. Here both move 16-byte vectors; reduce widens bf16 to binary32, adds in the
// order it is given (round to nearest even, no FMA: there is nothing to fuse), and rounds
// once back to bf16 with cvt.rn.
#pragma once

#include <stdint.h>

namespace coll {

// ------------------------------------------------------------------ memory ops (PTX)

// Read-only input data: non-coherent path, may be cached in L1.
__device__ __forceinline__ uint4 ld_nc_v4(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Streaming read (evict-first): data read exactly once.
__device__ __forceinline__ uint4 ld_cs_v4(const void *p) {
  uint4 r;
  asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Peer data written by another warp during this kernel: GPU-scope relaxed load, never
// served from a stale L1 line.
__device__ __forceinline__ uint4 ld_relaxed_v4(const void *p) {
  uint4 r;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p)
               : "memory");
  return r;
}

__device__ __forceinline__ void st_v4(void *p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Streaming store (evict-first): output written once.
__device__ __forceinline__ void st_cs_v4(void *p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long *p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void st_release_u32(uint32_t *p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Two 8-byte words, each single-copy atomic (tagged-data exchange).
__device__ __forceinline__ void st_relaxed_v2u64(void *p, unsigned long long a,
                                                 unsigned long long b) {
  asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1,%2};" ::"l"(p), "l"(a), "l"(b)
               : "memory");
}

__device__ __forceinline__ void ld_relaxed_v2u64(const void *p, unsigned long long &a,
                                                 unsigned long long &b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0,%1}, [%2];" : "=l"(a), "=l"(b) : "l"(p)
               : "memory");
}

__device__ __forceinline__ void st_relaxed_u32(uint32_t *p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_release_add_u32(uint32_t *p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ reduce arithmetic

// bf16x8 in a 16-byte vector -> 8 binary32 values (exact widening).
__device__ __forceinline__ void bf16x8_init(float a[8], uint4 v) {
  a[0] = __uint_as_float(v.x << 16);
  a[1] = __uint_as_float(v.x & 0xFFFF0000u);
  a[2] = __uint_as_float(v.y << 16);
  a[3] = __uint_as_float(v.y & 0xFFFF0000u);
  a[4] = __uint_as_float(v.z << 16);
  a[5] = __uint_as_float(v.z & 0xFFFF0000u);
  a[6] = __uint_as_float(v.w << 16);
  a[7] = __uint_as_float(v.w & 0xFFFF0000u);
}

__device__ __forceinline__ void bf16x8_add(float a[8], uint4 v) {
  a[0] = __fadd_rn(a[0], __uint_as_float(v.x << 16));
  a[1] = __fadd_rn(a[1], __uint_as_float(v.x & 0xFFFF0000u));
  a[2] = __fadd_rn(a[2], __uint_as_float(v.y << 16));
  a[3] = __fadd_rn(a[3], __uint_as_float(v.y & 0xFFFF0000u));
  a[4] = __fadd_rn(a[4], __uint_as_float(v.z << 16));
  a[5] = __fadd_rn(a[5], __uint_as_float(v.z & 0xFFFF0000u));
  a[6] = __fadd_rn(a[6], __uint_as_float(v.w << 16));
  a[7] = __fadd_rn(a[7], __uint_as_float(v.w & 0xFFFF0000u));
}

// Two binary32 -> packed bf16x2, round to nearest even (lo element in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint4 bf16x8_pack(const float a[8]) {
  return make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]),
                    pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7]));
}

__device__ __forceinline__ void f32x4_init(float a[4], uint4 v) {
  a[0] = __uint_as_float(v.x);
  a[1] = __uint_as_float(v.y);
  a[2] = __uint_as_float(v.z);
  a[3] = __uint_as_float(v.w);
}

__device__ __forceinline__ void f32x4_add(float a[4], uint4 v) {
  a[0] = __fadd_rn(a[0], __uint_as_float(v.x));
  a[1] = __fadd_rn(a[1], __uint_as_float(v.y));
  a[2] = __fadd_rn(a[2], __uint_as_float(v.z));
  a[3] = __fadd_rn(a[3], __uint_as_float(v.w));
}

__device__ __forceinline__ uint4 f32x4_pack(const float a[4]) {
  return make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                    __float_as_uint(a[3]));
}

// Accumulator over one 16-byte vector for element type DT (0 = bf16, 1 = f32).
template <int DT>
struct Vec16Acc {
  float a[DT == 0 ? 8 : 4];
  __device__ __forceinline__ void init(uint4 v) {
    if constexpr (DT == 0) bf16x8_init(a, v); else f32x4_init(a, v);
  }
  __device__ __forceinline__ void add(uint4 v) {
    if constexpr (DT == 0) bf16x8_add(a, v); else f32x4_add(a, v);
  }
  __device__ __forceinline__ uint4 pack() const {
    if constexpr (DT == 0) return bf16x8_pack(a); else return f32x4_pack(a);
  }
  __device__ __forceinline__ void addf(const Vec16Acc &o) {
#pragma unroll
    for (int i = 0; i < (DT == 0 ? 8 : 4); ++i) a[i] = __fadd_rn(a[i], o.a[i]);
  }
};

// Pairwise (tree) sum of the first kn (<= 8) vectors: ((x0+x1)+(x2+x3))+((x4+x5)+(x6+x7)),
// an unpaired element carried up a level. Accumulated into acc (which starts from this
// group's sum when `first`).
template <int DT>
__device__ __forceinline__ void tree8(Vec16Acc<DT> &acc, bool first, const uint4 x[8],
                                      uint32_t kn) {
  Vec16Acc<DT> p[4];
  const uint32_t np = (kn + 1) / 2;
#pragma unroll
  for (uint32_t i = 0; i < 4; ++i) {
    if (i < np) {
      p[i].init(x[2 * i]);
      if (2 * i + 1 < kn) p[i].add(x[2 * i + 1]);
    }
  }
  if (1 < np) p[0].addf(p[1]);
  if (3 < np) p[2].addf(p[3]);
  if (2 < np) p[0].addf(p[2]);
  if (first) acc = p[0]; else acc.addf(p[0]);
}

// ------------------------------------------------------------------ content tag

// Full-avalanche 32-bit mixer (two multiply / xor-shift rounds).
constexpr uint32_t kFmixK1 = 0x7FEB352Du, kFmixK2 = 0x846CA68Bu;
constexpr uint32_t kTagSalt = 0x9E3779B9u;
constexpr uint32_t kTagOff1 = 0x632BE5ABu, kTagOff2 = 0x165667B1u, kTagOff3 = 0xD3A2646Cu;
constexpr uint32_t kTagMulX = 0x85EBCA77u, kTagMulY = 0xC2B2AE3Du, kTagMulZ = 0x27D4EB2Fu,
                   kTagMulW = 0x9E3779B1u, kTagMulB = 0xA54FF53Bu;

__device__ __forceinline__ uint32_t fmix(uint32_t x) {
  x ^= x >> 16;
  x *= kFmixK1;
  x ^= x >> 15;
  x *= kFmixK2;
  x ^= x >> 16;
  return x;
}

// Contribution of vector `vi` (its index inside the piece) to the piece's two tags. Each
// word is salted by its position and multiplied by an odd constant (a bijection); tag A
// combines the four products with rotations and XOR and runs a full-avalanche round, tag B
// combines them with other rotations and additions and runs its own mixing round. The sums
// over vectors (lanes may be reduced in any order) then change with any change of the bytes
// except with probability about 2^-32 for tag A (which also catches structured changes such
// as two flipped sign bits) and 2^-48 for tag A with the 16 bits of tag B a flag keeps.
__device__ __forceinline__ uint2 tag_part(uint4 v, uint32_t vi) {
  const uint32_t s = vi * kTagSalt;
  const uint32_t a = (v.x ^ s) * kTagMulX;
  const uint32_t b = (v.y ^ (s + kTagOff1)) * kTagMulY;
  const uint32_t c = (v.z ^ (s + kTagOff2)) * kTagMulZ;
  const uint32_t d = (v.w ^ (s + kTagOff3)) * kTagMulW;
  const uint32_t ta = fmix(a ^ __funnelshift_l(b, b, 8) ^ __funnelshift_l(c, c, 16) ^
                           __funnelshift_l(d, d, 24));
  uint32_t tb = a + __funnelshift_l(b, b, 13) + __funnelshift_l(c, c, 7) +
                __funnelshift_l(d, d, 21);
  tb ^= tb >> 16;
  tb *= kTagMulB;
  tb ^= tb >> 13;
  return make_uint2(ta, tb);
}

// The sums of tag_part(v[k], vi) over k < kn, the same values, computed stage by stage: the
// eight vectors' independent dependency chains then interleave on the one warp that
// validates a piece (computed one after the other they cost about twice as long).
__device__ __forceinline__ uint2 tag_parts8(const uint4 v[8], uint32_t kn, uint32_t vi) {
  const uint32_t s = vi * kTagSalt;
  uint32_t t[8], u[8];
#pragma unroll
  for (uint32_t k = 0; k < 8; ++k) {
    t[k] = (v[k].x ^ s) * kTagMulX;
    u[k] = t[k];
  }
#pragma unroll
  for (uint32_t k = 0; k < 8; ++k) {
    const uint32_t b = (v[k].y ^ (s + kTagOff1)) * kTagMulY;
    t[k] ^= __funnelshift_l(b, b, 8);
    u[k] += __funnelshift_l(b, b, 13);
  }
#pragma unroll
  for (uint32_t k = 0; k < 8; ++k) {
    const uint32_t c = (v[k].z ^ (s + kTagOff2)) * kTagMulZ;
    t[k] ^= __funnelshift_l(c, c, 16);
    u[k] += __funnelshift_l(c, c, 7);
  }
#pragma unroll
  for (uint32_t k = 0; k < 8; ++k) {
    const uint32_t d = (v[k].w ^ (s + kTagOff3)) * kTagMulW;
    t[k] ^= __funnelshift_l(d, d, 24);
    u[k] += __funnelshift_l(d, d, 21);
  }
#pragma unroll
  for (uint32_t k = 0; k < 8; ++k) {
    t[k] ^= t[k] >> 16;
    u[k] ^= u[k] >> 16;
  }
#pragma unroll
  for (uint32_t k = 0; k < 8; ++k) {
    t[k] *= kFmixK1;
    u[k] *= kTagMulB;
  }
#pragma unroll
  for (uint32_t k = 0; k < 8; ++k) {
    t[k] ^= t[k] >> 15;
    u[k] ^= u[k] >> 13;
  }
#pragma unroll
  for (uint32_t k = 0; k < 8; ++k) t[k] *= kFmixK2;
#pragma unroll
  for (uint32_t k = 0; k < 8; ++k) t[k] ^= t[k] >> 16;
  uint2 h = make_uint2(0u, 0u);
#pragma unroll
  for (uint32_t k = 0; k < 8; ++k)
    if (k < kn) {
      h.x += t[k];
      h.y += u[k];
    }
  return h;
}

// A piece's tag: its hash plus the epoch times an odd constant (linear, so that tags of
// several producers can be checked as one sum).
__device__ __forceinline__ uint32_t tag_fold(uint32_t h, uint32_t epoch) {
  return h + epoch * 0x85EBCA6Bu;
}
__device__ __forceinline__ uint32_t tag_fold_b(uint32_t h, uint32_t epoch) {
  return h + epoch * 0xC2B2AE35u;
}
__device__ __forceinline__ uint2 reduce_add2(uint2 h) {
  return make_uint2(__reduce_add_sync(0xFFFFFFFFu, h.x), __reduce_add_sync(0xFFFFFFFFu, h.y));
}

}  // namespace coll
