// Device-side helpers shared by the kernels of libcsa: error word, paging,
// RoPE angles and the storage codecs (bf16, e4m3, e2m1).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "csa.h"

namespace csa {

constexpr int kMaxRopePairs = 64;  // rope_dim <= 128

// Rotary frequencies as turn fractions: turns[k] = round(2^64 * theta^(-2k/r) / (2 pi)),
// filled on the host in double.  The angle of position p is then
// (p * turns[k] mod 2^64) / 2^64 turns: one exact wrapping 64-bit integer
// multiply gives the reduced angle, with an error of about p * 2^-53 turns,
// far below a microradian at p ~ 2^20 (an fp32 product would be off by 0.06 rad).
struct RopeTab {
  uint64_t turns[kMaxRopePairs];
  int32_t rope_dim;
};

// Programmatic dependent launch.  Every kernel of the library is launched so
// that it may start while the previous kernel of the stream (the library's or
// anyone's) is finishing: pdl_trigger() lets the next kernel launch;
// pdl_wait() blocks until the previous kernel has completed and its writes
// are visible.  Every kernel calls pdl_wait() before its first access to
// global memory -- only set-up that touches no memory (barrier init, TMEM
// allocation) runs before it -- so a kernel is ordered after all work
// enqueued before it exactly as in plain stream order, and every CTA passes
// pdl_wait() before it exits, so completion stays transitive along the stream.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void record_error(int32_t* err, int32_t code) {
  if (err) atomicCAS(err, 0, code);
}

// Physical row of logical row `lrow` of sequence `seq`, or -1 (and the error
// word set) when the table or the cache has no such row.
__device__ __forceinline__ int64_t phys_row(const csa_block_table& bt, const csa_paged& c, int seq,
                                            int64_t lrow, int32_t* err) {
  if (seq < 0 || seq >= bt.num_seqs || lrow < 0) {
    record_error(err, CSA_ERR_DEVICE_BOUNDS);
    return -1;
  }
  int64_t lb = lrow / c.rows_per_block;
  if (lb >= bt.stride) {
    record_error(err, CSA_ERR_DEVICE_BOUNDS);
    return -1;
  }
  int32_t pb = bt.table[(int64_t)seq * bt.stride + lb];
  if (pb < 0 || pb >= c.num_blocks) {
    record_error(err, CSA_ERR_DEVICE_BOUNDS);
    return -1;
  }
  return (int64_t)pb * c.rows_per_block + (lrow - lb * c.rows_per_block);
}

// Bytes of one row of a paged cache (see csa_paged in csa.h).
__host__ __device__ __forceinline__ int64_t row_bytes(const csa_paged& c) {
  switch (c.dtype) {
    case CSA_F32: return (int64_t)c.dim * 4;
    case CSA_BF16: return (int64_t)c.dim * 2;
    case CSA_E4M3: return c.dim;
    case CSA_E4M3R: return (int64_t)c.dim + c.tail_bf16;
    default: return c.dim / 2;  // CSA_E2M1
  }
}

// Number of compressed entries visible to a query at p: entries whose last raw
// token ratio*i+window-1 lies before p.
__host__ __device__ __forceinline__ int32_t n_visible(int32_t p, int32_t ratio, int32_t window) {
  return p < window ? 0 : (p - window) / ratio + 1;
}

// cos / sin of the rotary angle of pair k at position pos, reduced to [-pi, pi).
// Only the top 32 bits of the wrapped 64-bit product are needed (an angle
// step of 2 pi / 2^32), and they come from 32-bit integer multiplies.
__device__ __forceinline__ void rope_cs(const RopeTab& t, int k, int64_t pos, float& c, float& s) {
  const uint32_t p = (uint32_t)pos;
  const uint64_t f = t.turns[k];
  const uint32_t lo_hi = __umulhi(p, (uint32_t)f);           // bits 32..63 of p * f_lo
  const uint32_t top = lo_hi + p * (uint32_t)(f >> 32);      // bits 32..63 of p * f, mod 2^32
  const float a = (float)(int32_t)top * 1.4629180792671596e-9f;  // 2 pi / 2^32
  sincosf(a, &s, &c);
}

// ---------------------------------------------------------------- codecs

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16(float x) {
  __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&h);
}

// Two floats rounded to bf16 (nearest even) in one instruction: lo in bits 0..15, hi in 16..31.
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// e4m3 (fn): sign | 4 exponent bits (bias 7) | 3 mantissa bits; exponent 0 is
// subnormal (m * 2^-9); 0x7f / 0xff are NaN.
__device__ __forceinline__ float e4m3_to_f32(uint8_t v) {
  uint32_t s = (uint32_t)(v & 0x80) << 24;
  uint32_t e = (v >> 3) & 0xF;
  uint32_t m = v & 0x7;
  if (e == 0) {
    float f = (float)m * 0.001953125f;  // 2^-9
    return __uint_as_float(__float_as_uint(f) | s);
  }
  if (e == 0xF && m == 0x7) return __uint_as_float(0x7FC00000u | s);
  return __uint_as_float(s | ((e + 120u) << 23) | (m << 20));
}

// Two e4m3 codes (bits 0-7: lo, 8-15: hi) to two floats through the hardware
// e4m3x2 -> f16x2 conversion, exact (every e4m3 value is an f16 value).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two) {
  uint32_t h2;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h2) : "r"(two));
  float lo, hi;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h2));
  return make_float2(lo, hi);
}

// Round-to-nearest-even to e4m3 with saturation to +-448 (hardware cvt).
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;  // lo in bits 0..7, hi in bits 8..15
}

__device__ __forceinline__ uint8_t f32_to_e4m3(float x) {
  return (uint8_t)(f32x2_to_e4m3x2(x, 0.0f) & 0xFF);
}

// e2m1: sign | 2 exponent bits (bias 1) | 1 mantissa bit; magnitudes
// 0, 0.5, 1, 1.5, 2, 3, 4, 6.
__device__ __forceinline__ float e2m1_to_f32(uint32_t c) {
  // magnitude code m: exponent bits m>>1 (bias 1), mantissa bit m&1; exponent 0
  // is the subnormal 0 / 0.5.  Built as fp32 bits (no table, no local memory).
  const uint32_t m = c & 7;
  const uint32_t mag = m >= 2 ? (((m >> 1) + 126u) << 23) | ((m & 1u) << 22) : (m ? 0x3F000000u : 0u);
  return __uint_as_float(mag | ((c & 8u) << 28));
}

// Nearest e2m1 code, ties to the even code, saturating at 6.  Decision points
// are the midpoints between neighbours; a midpoint goes to the neighbour whose
// mantissa bit is 0.
__device__ __forceinline__ uint32_t f32_to_e2m1(float x) {
  float a = fabsf(x);
  uint32_t m;
  if (a <= 0.25f) m = 0;
  else if (a < 0.75f) m = 1;
  else if (a <= 1.25f) m = 2;
  else if (a < 1.75f) m = 3;
  else if (a <= 2.5f) m = 4;
  else if (a < 3.5f) m = 5;
  else if (a <= 5.0f) m = 6;
  else m = 7;
  return m | (signbit(x) ? 8u : 0u);
}

// One group of 16 values -> 8 bytes of e2m1 codes (element e in nibble e of the
// little-endian pair of words: element 2j in the low nibble of byte j) and the
// group's e4m3 scale byte: scale = e4m3_rn(amax/6); code = e2m1_rn(v / scale);
// a zero scale gives zero codes.  `v` may point to shared or local memory.
__device__ __forceinline__ uint8_t quantize_e2m1_group(const float* v, uint2& packed) {
  float am = 0.f;
#pragma unroll
  for (int e = 0; e < 16; ++e) am = fmaxf(am, fabsf(v[e]));
  const uint8_t sc = f32_to_e4m3(am / 6.0f);
  const float s = e4m3_to_f32(sc);
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const uint32_t code = s > 0.f ? f32_to_e2m1(v[e] / s) : 0u;
    w[e / 8] |= code << (4 * (e % 8));
  }
  packed = make_uint2(w[0], w[1]);
  return sc;
}

// ---------------------------------------------------------------- reductions

// 2^x with the special-function unit (about 2 ulp); the softmax weights need no more.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

// Block-wide sum / max; `red` is shared scratch of >= 32 floats.  All threads
// of the block must call it; blockDim.x is a multiple of 32.
__device__ __forceinline__ float block_sum(float v, float* red) {
  int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : 0.f;
  return warp_sum(t);
}

__device__ __forceinline__ float block_max(float v, float* red) {
  int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : 0.f;
  return warp_max(t);
}

// ---------------------------------------------------------------- row access

// Element e of a row of a F32 / BF16 cache, or of an input array.
__device__ __forceinline__ float load_elem(const void* base, int32_t dtype, int64_t idx) {
  if (dtype == CSA_F32) return reinterpret_cast<const float*>(base)[idx];
  return bf16_to_f32(reinterpret_cast<const uint16_t*>(base)[idx]);
}

}  // namespace csa
