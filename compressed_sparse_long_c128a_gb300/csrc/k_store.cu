// Quantising row insert into a paged cache (indexer-key insert, loading held entries).
//
// Pages: "vLLM解密：DeepSeek-V4本地部署為何如此困難" §3.2 first fusion (the
// indexer K cache has its own insert kernel); "vLLM DeepSeek V4 Support",
// "DeepSeek V4 Attention Architecture" last paragraph (fp4 indexer cache, fp8
// attention cache).
//   E4M3: scale = amax/448 per row; code = e4m3_rn_satfinite(x * (448/amax)).
//   E4M3R: the same over the first dim - tail_bf16 elements; the tail in bf16.
//   E2M1: per 16 elements, scale = e4m3_rn(amax16/6); code = e2m1_rn(x / scale).

#include "csa_kernels.h"

namespace csa {
namespace {

constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads) store_kernel(const StoreArgs a) {
  __shared__ float red[32];
  pdl_trigger();
  pdl_wait();
  const int j = blockIdx.x;
  const csa_paged& c = a.cache;
  const int D = c.dim;
  const int64_t prow = phys_row(a.bt, c, a.seq_id[j], a.row_idx[j], a.err);
  if (prow < 0) return;  // block-uniform
  const float* x = a.rows + (int64_t)j * D;

  if (c.dtype == CSA_F32) {
    float* row = reinterpret_cast<float*>(c.data) + prow * D;
    for (int d = threadIdx.x; d < D; d += blockDim.x) row[d] = x[d];
  } else if (c.dtype == CSA_BF16) {
    uint16_t* row = reinterpret_cast<uint16_t*>(c.data) + prow * D;
    for (int d = threadIdx.x; d < D; d += blockDim.x) row[d] = f32_to_bf16(x[d]);
  } else if (c.dtype == CSA_E4M3 || c.dtype == CSA_E4M3R) {
    // e4m3 codes + per-row scale over [0, Dq); an E4M3R row keeps [Dq, D) in bf16
    const int Dq = c.dtype == CSA_E4M3R ? D - c.tail_bf16 : D;
    float am = 0.f;
    for (int d = threadIdx.x; d < Dq; d += blockDim.x) am = fmaxf(am, fabsf(x[d]));
    am = block_max(am, red);
    const float inv = am > 0.f ? 448.0f / am : 0.0f;
    uint8_t* row = reinterpret_cast<uint8_t*>(c.data) + prow * row_bytes(c);
    for (int pr = threadIdx.x; pr < Dq / 2; pr += blockDim.x)
      *reinterpret_cast<uint16_t*>(row + 2 * pr) = f32x2_to_e4m3x2(x[2 * pr] * inv, x[2 * pr + 1] * inv);
    for (int pr = threadIdx.x; pr < (D - Dq) / 2; pr += blockDim.x)
      *reinterpret_cast<uint32_t*>(row + Dq + 4 * pr) = f32x2_to_bf16x2(x[Dq + 2 * pr], x[Dq + 2 * pr + 1]);
    if (threadIdx.x == 0) reinterpret_cast<float*>(c.scales)[prow] = am / 448.0f;
  } else {  // E2M1, one thread per group of 16
    uint8_t* row = reinterpret_cast<uint8_t*>(c.data) + prow * (D / 2);
    uint8_t* srow = reinterpret_cast<uint8_t*>(c.scales) + prow * (D / 16);
    for (int g = threadIdx.x; g < D / 16; g += blockDim.x) {
      float v[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = x[g * 16 + e];
      uint2 packed;
      srow[g] = quantize_e2m1_group(v, packed);
      *reinterpret_cast<uint2*>(row + g * 8) = packed;
    }
  }
}

}  // namespace

cudaError_t launch_store(const StoreArgs& a, int32_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  return launch_k(store_kernel, dim3(n), dim3(kThreads), 0, s, 0, a);
}

}  // namespace csa
