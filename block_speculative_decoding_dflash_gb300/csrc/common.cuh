// Device helpers shared by the libdflash kernels: storage types, vector
// loads, warp reductions, and the device-resident state of a ring and of a
// round.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dfl {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------------------
// Device-resident state. Kept in device memory so that whole rounds can be
// enqueued (and graph-captured) without the host reading anything back.
// ---------------------------------------------------------------------------
struct RingState {
  long long offset;    // next absolute position to be written
  long long base;      // oldest position written since the last reset
  long long hw;        // highest position ever written (high-water mark)
  int appended;        // rows appended since the last trim / commit
  int error;           // sticky error bits (kErr*)
};

struct RoundState {
  int anchor;          // current anchor token
  int n;               // last verify: accepted + 1
  int a;               // last verify: accepted
  int bonus;           // last verify: t_a
  int block;           // width of the last draft
  int error;           // sticky error bits (kErr*)
  long long rounds;    // committed rounds
  long long proposed;  // sum of block - 1
  long long accepted;  // sum of a
  long long emitted;   // sum of a + 1
};

enum : int {
  kErrFull = 1,        // append-only ring overflow (rows skipped)
  kErrRange = 2,       // a token id outside the vocabulary reached a gather
  kErrTrim = 16,       // a target trim longer than the rows appended since the last one
  kErrPos = 8,         // a draft's host-given anchor position was not the
                       // committed context length
};

// ---------------------------------------------------------------------------
// Storage conversions. Accumulation is always fp32; a value is rounded to the
// storage type exactly where it is stored.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

template <typename T> __device__ __forceinline__ float rnd(float x) { return to_f(from_f<T>(x)); }

// Exact bf16 -> fp32 of the two halves of a 32-bit word.
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Streaming 16-byte load that does not allocate in L1 (weights are read once).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// 8 consecutive elements as fp32; p must be 16-byte aligned.
__device__ __forceinline__ void load8(const bf16* p, float* o) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  o[0] = bf_lo(u.x); o[1] = bf_hi(u.x); o[2] = bf_lo(u.y); o[3] = bf_hi(u.y);
  o[4] = bf_lo(u.z); o[5] = bf_hi(u.z); o[6] = bf_lo(u.w); o[7] = bf_hi(u.w);
}
__device__ __forceinline__ void load8(const float* p, float* o) {
  float4 a = reinterpret_cast<const float4*>(p)[0];
  float4 b = reinterpret_cast<const float4*>(p)[1];
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
  o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
__device__ __forceinline__ void load8_stream(const bf16* p, float* o) {
  uint4 u = ld_stream(p);
  o[0] = bf_lo(u.x); o[1] = bf_hi(u.x); o[2] = bf_lo(u.y); o[3] = bf_hi(u.y);
  o[4] = bf_lo(u.z); o[5] = bf_hi(u.z); o[6] = bf_lo(u.w); o[7] = bf_hi(u.w);
}
__device__ __forceinline__ void load8_stream(const float* p, float* o) {
  uint4 a = ld_stream(p);
  uint4 b = ld_stream(p + 4);
  o[0] = __uint_as_float(a.x); o[1] = __uint_as_float(a.y);
  o[2] = __uint_as_float(a.z); o[3] = __uint_as_float(a.w);
  o[4] = __uint_as_float(b.x); o[5] = __uint_as_float(b.y);
  o[6] = __uint_as_float(b.z); o[7] = __uint_as_float(b.w);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// (value, index) argmax step: the larger value wins and equal values keep the
// lower index. The rule does not depend on the order of comparisons, so any
// reduction tree gives the same answer.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, v, o);
    int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (better(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

__device__ __forceinline__ long long ring_slot(long long pos, long long cap) {
  return pos % cap;
}

// Optional per-launch timeline (globaltimer, ns): a launch owns slot `slot` of
// three arrays: [0] earliest CTA entry (min), [1] latest return from the
// programmatic-dependency wait (max), [2] latest CTA exit (max).
struct KTrace {
  unsigned long long* p;   // [3][kTraceSlots] or NULL
  int slot;
};
constexpr int kKTraceSlots = 256;
__device__ __forceinline__ unsigned long long ktrace_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Call from one thread per CTA.
__device__ __forceinline__ void ktrace_mark(const KTrace& t, int k) {
  if (!t.p) return;
  unsigned long long* a = t.p + (size_t)k * kKTraceSlots + t.slot;
  if (k == 0) atomicMin(a, ktrace_now());
  else atomicMax(a, ktrace_now());
}

// (cos, sin) of pos * inv_freq[i]; the angle is formed in fp64 so that large
// absolute positions keep their precision.
__device__ __forceinline__ float2 rope_entry(const double* inv_freq, int i, long long pos) {
  double s, c;
  sincos(static_cast<double>(pos) * inv_freq[i], &s, &c);
  return make_float2(static_cast<float>(c), static_cast<float>(s));
}

}  // namespace dfl
