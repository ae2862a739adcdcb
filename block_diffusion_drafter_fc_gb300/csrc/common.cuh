// Device helpers shared by the drafter kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define DF_DEVICE __device__ __forceinline__

namespace dflash {

constexpr int kBlock = 16;       // rows of one noise block
constexpr int kWarp = 32;

// ---------------------------------------------------------------- conversions

DF_DEVICE float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// Round an fp32 value to bf16 bits, nearest-even (the hardware conversion).
DF_DEVICE uint16_t f32_to_bf16_bits(float x) {
  __nv_bfloat16 b = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&b);
}

// Pack two fp32 values into a bf16x2 register (low half = first element).
DF_DEVICE uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Split fp32 pairs into bf16 hi + bf16 lo parts: x = hi + lo + O(2^-17 |x|).
DF_DEVICE void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  float2 hf = __bfloat1622float2(h);
  __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = *reinterpret_cast<uint32_t*>(&l);
}

// Split fp32 pairs into fp16 hi + fp16 lo parts (the activation pair of FP4
// weights, whose products run in fp16): x = hi + lo to 2^-22 |x| (2^-25 absolute
// below 2^-3); |x| must stay below 65504.
DF_DEVICE void split_f16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// The 16-bit activation pair of a projection input: bf16, or fp16 with FP4 weights.
DF_DEVICE void split_pair16x2(float a, float b, bool f16, uint32_t& hi, uint32_t& lo) {
  if (f16)
    split_f16x2(a, b, hi, lo);
  else
    split_bf16x2(a, b, hi, lo);
}
DF_DEVICE void split_pair16(float x, bool f16, uint16_t& hi, uint16_t& lo) {
  uint32_t h, l;
  split_pair16x2(x, 0.f, f16, h, l);
  hi = (uint16_t)(h & 0xffffu);
  lo = (uint16_t)(l & 0xffffu);
}

// Two E4M3 codes (low byte = first element) -> bf16x2.  Every E4M3 value is
// exact in fp16 and in bf16, so the two hardware conversions lose nothing.
DF_DEVICE uint32_t e4m3x2_to_bf16x2(uint16_t v) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
  float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
  return pack_bf16x2(f.x, f.y);
}

// Two E4M3 codes (low byte = first element) -> f16x2, exact: one conversion.
DF_DEVICE uint32_t e4m3x2_to_f16x2(uint16_t v) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

DF_DEVICE float e4m3_to_f32(uint8_t v) {
  __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(v), __NV_E4M3);
  return __half2float(*reinterpret_cast<__half*>(&h));
}

// Load element i of a dense (f32 or bf16) vector/matrix as fp32.
DF_DEVICE float load_dense(const void* p, int dtype_bf16, size_t i) {
  return dtype_bf16 ? bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(p)[i])
                    : reinterpret_cast<const float*>(p)[i];
}

// ---------------------------------------------------------------- reductions

DF_DEVICE float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

DF_DEVICE float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// (value, index) argmax with the lowest index on ties; NaN never wins.
DF_DEVICE void argmax_merge(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) { v = v2; i = i2; }
}

DF_DEVICE void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    argmax_merge(v, i, v2, i2);
  }
}

// ---------------------------------------------------------------- memory

// 16-byte streaming load that bypasses L1 allocation (weights are read once).
DF_DEVICE uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Bulk prefetch of a contiguous global range into L2 (no registers, no shared
// memory); address 16-byte aligned, size a multiple of 16.
DF_DEVICE void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- dependent launch

// Programmatic dependent launch: let the next kernel of the stream be scheduled
// now (it only starts where this grid frees resources), and, before reading
// anything an earlier kernel wrote, wait until the preceding grid has completed
// and its memory is visible.  Only immutable data (weights) is touched before
// the wait.  Both are no-ops for a kernel launched without the attribute.
DF_DEVICE void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
DF_DEVICE void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- launch timestamps

// Per-launch timing inside a replayed graph (profiling captures only; a null
// slot records nothing).  Slot s: s[0] = ~(earliest CTA start), s[1] = latest
// CTA end, both %globaltimer nanoseconds, so one zero fill resets a slot and
// both updates are atomicMax.  One thread per CTA calls each.
DF_DEVICE unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
DF_DEVICE void stamp_begin(unsigned long long* s) {
  if (s) atomicMax(s, ~global_ns());
}
DF_DEVICE void stamp_finish(unsigned long long* s) {
  if (s) atomicMax(s + 1, global_ns());
}

// ---------------------------------------------------------------- tensor cores

// D += A * B for one m16n8k16 bf16 tile with fp32 accumulation.
DF_DEVICE void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D += A * B for one m16n8k16 fp16 tile with fp32 accumulation.
DF_DEVICE void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

}  // namespace dflash
