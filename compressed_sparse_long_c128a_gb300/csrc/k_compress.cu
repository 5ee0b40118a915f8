// Compressor + RMSNorm + RoPE + cache insert, and the raw sliding-window insert.
//
// Pages ("vLLM解密：DeepSeek-V4本地部署為何如此困難" §3.2, first and third
// fusion; "vLLM DeepSeek V4 Support", "KV Cache Memory Management" item 2):
// the compressed key is normalised, rotated and written to the cache in one
// elementwise kernel, and the compressor's rolling residual lives in a
// sliding-window style state cache.  Here that is two launches: `ingest`
// writes each new token's state row and window row; `emit` then forms every
// entry whose window closed at one of the tokens, reading the window's raw rows
// back from the state cache (so a window may span earlier calls).

#include "csa_kernels.h"

namespace csa {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void store_elem(void* base, int32_t dtype, int64_t idx, float v) {
  if (dtype == CSA_F32)
    reinterpret_cast<float*>(base)[idx] = v;
  else
    reinterpret_cast<uint16_t*>(base)[idx] = f32_to_bf16(v);
}

// Write y[0..D) (shared memory) as physical row `prow` of cache c.  Called by
// the whole block with a block-uniform prow >= 0.
__device__ void store_row(const csa_paged& c, int64_t prow, const float* y, int D, float* red) {
  if (c.dtype == CSA_E4M3) {
    float am = 0.f;
    for (int d = threadIdx.x; d < D; d += blockDim.x) am = fmaxf(am, fabsf(y[d]));
    am = block_max(am, red);
    const float scale = am / 448.0f;
    const float inv = am > 0.f ? 448.0f / am : 0.0f;
    uint8_t* row = reinterpret_cast<uint8_t*>(c.data) + prow * (int64_t)D;
    for (int pr = threadIdx.x; pr < D / 2; pr += blockDim.x)
      *reinterpret_cast<uint16_t*>(row + 2 * pr) = f32x2_to_e4m3x2(y[2 * pr] * inv, y[2 * pr + 1] * inv);
    if (threadIdx.x == 0) reinterpret_cast<float*>(c.scales)[prow] = scale;
  } else if (c.dtype == CSA_E2M1) {  // one thread per group of 16 (D % 16 == 0)
    uint8_t* row = reinterpret_cast<uint8_t*>(c.data) + prow * (int64_t)(D / 2);
    uint8_t* srow = reinterpret_cast<uint8_t*>(c.scales) + prow * (int64_t)(D / 16);
    for (int g = threadIdx.x; g < D / 16; g += blockDim.x) {
      uint2 packed;
      srow[g] = quantize_e2m1_group(y + 16 * g, packed);
      *reinterpret_cast<uint2*>(row + g * 8) = packed;
    }
  } else if (c.dtype == CSA_BF16) {
    uint16_t* row = reinterpret_cast<uint16_t*>(c.data) + prow * (int64_t)D;
    for (int pr = threadIdx.x; pr < D / 2; pr += blockDim.x) {
      uint32_t v = (uint32_t)f32_to_bf16(y[2 * pr]) | ((uint32_t)f32_to_bf16(y[2 * pr + 1]) << 16);
      *reinterpret_cast<uint32_t*>(row + 2 * pr) = v;
    }
  } else {
    float* row = reinterpret_cast<float*>(c.data) + prow * (int64_t)D;
    for (int pr = threadIdx.x; pr < D / 2; pr += blockDim.x)
      *reinterpret_cast<float2*>(row + 2 * pr) = make_float2(y[2 * pr], y[2 * pr + 1]);
  }
}

// y := RoPE(y * inv_rms * gamma, pos) in place, pairs (2k, 2k+1) over the last r dims.
__device__ void norm_rope_inplace(float* y, int D, float inv_rms, const float* gamma, const RopeTab& rt,
                                  int64_t pos) {
  const int R = rt.rope_dim;
  for (int pr = threadIdx.x; pr < D / 2; pr += blockDim.x) {
    int d = 2 * pr;
    float y0 = y[d] * inv_rms * gamma[d];
    float y1 = y[d + 1] * inv_rms * gamma[d + 1];
    if (d >= D - R) {
      float c, s;
      rope_cs(rt, (d - (D - R)) / 2, pos, c, s);
      float t0 = y0 * c - y1 * s;
      y1 = y0 * s + y1 * c;
      y0 = t0;
    }
    y[d] = y0;
    y[d + 1] = y1;
  }
}

__global__ void __launch_bounds__(kThreads) ingest_kernel(const IngestArgs a) {
  extern __shared__ float y[];
  __shared__ float red[32];
  pdl_trigger();
  pdl_wait();
  const int j = blockIdx.x;
  const int D = a.dim;
  const int seq = a.seq_id[j];
  const int64_t p = a.pos[j];
  const int64_t srow = phys_row(a.state_bt, a.state, seq, p, a.err);
  const int64_t wrow = a.swa.data ? phys_row(a.swa_bt, a.swa, seq, p, a.err) : -1;  // no window cache: state only

  float ss = 0.f;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float x = load_elem(a.kv, a.in_dtype, (int64_t)j * D + d);
    y[d] = x;
    ss += x * x;
    if (srow >= 0) {
      float g = load_elem(a.gate, a.in_dtype, (int64_t)j * D + d);
      store_elem(a.state.data, a.state.dtype, srow * 2 * D + d, x);
      store_elem(a.state.data, a.state.dtype, srow * 2 * D + D + d, g);
    }
  }
  ss = block_sum(ss, red);
  if (wrow < 0) return;  // block-uniform
  const float inv = 1.0f / sqrtf(ss / (float)D + a.eps);
  __syncthreads();
  norm_rope_inplace(y, D, inv, a.gamma_swa, a.rope, p);
  __syncthreads();
  store_row(a.swa, wrow, y, D, red);
}

__global__ void __launch_bounds__(kThreads) emit_kernel(const EmitArgs a) {
  extern __shared__ float y[];
  __shared__ float red[32];
  __shared__ int64_t rows[256];
  __shared__ int bad;
  const int j = blockIdx.x;
  const int64_t t = a.pos[j];
  const int W = a.window, Rt = a.ratio, D = a.dim;
  pdl_trigger();
  // every CTA waits, even one with nothing to emit: this grid may only complete
  // after the ingest launch has, so later launches that wait on this one also
  // see ingest's writes
  pdl_wait();
  if (t < W - 1 || (t - W + 1) % Rt) return;  // no window closes at this token
  const int64_t i = (t - W + 1) / Rt;
  const int64_t base = i * Rt;  // first raw position = anchor
  const int seq = a.seq_id[j];

  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  for (int o = threadIdx.x; o < W; o += blockDim.x) {
    int64_t r = phys_row(a.state_bt, a.state, seq, base + o, a.err);
    rows[o] = r;
    if (r < 0) bad = 1;
  }
  const int64_t crow = phys_row(a.comp_bt, a.comp, seq, i, a.err);
  __syncthreads();
  if (bad || crow < 0) return;

  const int sdt = a.state.dtype;
  float ss = 0.f;
  for (int pr = threadIdx.x; pr < D / 2; pr += blockDim.x) {
    const int d = 2 * pr;
    float m0 = -INFINITY, m1 = -INFINITY, s0 = 0.f, s1 = 0.f, c0 = 0.f, c1 = 0.f;
#pragma unroll 4
    for (int o = 0; o < W; ++o) {
      const int64_t rb = rows[o] * 2 * D;
      const float k0 = load_elem(a.state.data, sdt, rb + d);
      const float k1 = load_elem(a.state.data, sdt, rb + d + 1);
      const float g0 = load_elem(a.state.data, sdt, rb + D + d) + a.bias[o * D + d];
      const float g1 = load_elem(a.state.data, sdt, rb + D + d + 1) + a.bias[o * D + d + 1];
      // online softmax over the window offsets, per channel
      if (g0 > m0) {
        const float f = expf(m0 - g0);
        s0 = s0 * f + 1.f;
        c0 = c0 * f + k0;
        m0 = g0;
      } else {
        const float e = expf(g0 - m0);
        s0 += e;
        c0 += e * k0;
      }
      if (g1 > m1) {
        const float f = expf(m1 - g1);
        s1 = s1 * f + 1.f;
        c1 = c1 * f + k1;
        m1 = g1;
      } else {
        const float e = expf(g1 - m1);
        s1 += e;
        c1 += e * k1;
      }
    }
    const float v0 = c0 / s0, v1 = c1 / s1;
    y[d] = v0;
    y[d + 1] = v1;
    ss += v0 * v0 + v1 * v1;
  }
  ss = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / (float)D + a.eps);
  __syncthreads();
  norm_rope_inplace(y, D, inv, a.gamma_c, a.rope, base);
  __syncthreads();
  store_row(a.comp, crow, y, D, red);
}

}  // namespace

cudaError_t launch_ingest(const IngestArgs& a, int32_t n_tok, cudaStream_t s) {
  if (n_tok == 0) return cudaSuccess;
  return launch_k(ingest_kernel, dim3(n_tok), dim3(kThreads), a.dim * sizeof(float), s, kStreamOrder, 0, a);
}

cudaError_t launch_emit(const EmitArgs& a, int32_t n_tok, cudaStream_t s) {
  if (n_tok == 0) return cudaSuccess;
  return launch_k(emit_kernel, dim3(n_tok), dim3(kThreads), a.dim * sizeof(float), s, kAfterOwnKernel, 0, a);
}

}  // namespace csa
