// DSA indexer scores: s_i = sum_h w_h * relu(q_idx_h . key_i) over the
// entries visible to each query row ("vLLM解密：DeepSeek-V4本地部署為何如此困難"
// §二 item 3; "vLLM DeepSeek V4 Support", "DeepSeek Sparse Attention (DSA)").
//
// Generic CUDA-core path: any head count / dim, keys in F32, BF16 or E2M1.
// One CTA takes one query row and a strided set of 64-entry tiles; the
// row's query heads sit in shared memory as fp32, each tile of keys is
// dequantised into shared memory, and thread (entry e, head quarter hq) adds
// w_h * relu(dot) over its quarter of the heads.

#include "csa_kernels.h"

namespace csa {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 64;  // entries per tile
constexpr int kQuarters = kThreads / kTile;

__device__ __forceinline__ float key_elem(const csa_paged& c, int64_t prow, int d) {
  if (c.dtype == CSA_F32) return reinterpret_cast<const float*>(c.data)[prow * c.dim + d];
  if (c.dtype == CSA_BF16) return bf16_to_f32(reinterpret_cast<const uint16_t*>(c.data)[prow * c.dim + d]);
  const uint8_t b = reinterpret_cast<const uint8_t*>(c.data)[prow * (c.dim / 2) + d / 2];
  const uint8_t sc = reinterpret_cast<const uint8_t*>(c.scales)[prow * (c.dim / 16) + d / 16];
  return e2m1_to_f32((d & 1) ? (b >> 4) : (b & 0xF)) * e4m3_to_f32(sc);
}

__global__ void __launch_bounds__(kThreads) indexer_scores_kernel(const IndexerArgs a) {
  extern __shared__ float smem[];
  const int H = a.heads, Dk = a.dim, ld = Dk + 1;
  float* qs = smem;                  // [H][Dk]
  float* ws = qs + H * Dk;           // [H]
  float* ks = ws + H;                // [kTile][Dk+1]
  float* part = ks + kTile * ld;     // [kQuarters][kTile]
  __shared__ int64_t prow_s[kTile];

  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  const int32_t p = a.pos[r];
  const int seq = a.seq_id[r];
  const int32_t n = n_visible(p, a.ratio, a.window);
  if (n > a.max_n) {
    if (threadIdx.x == 0) record_error(a.err, CSA_ERR_DEVICE_BOUNDS);
    return;
  }
  for (int x = threadIdx.x; x < H * Dk; x += blockDim.x)
    qs[x] = load_elem(a.q_idx, a.q_dtype, (int64_t)r * H * Dk + x);
  for (int x = threadIdx.x; x < H; x += blockDim.x) ws[x] = a.w[(int64_t)r * H + x];

  const int e = threadIdx.x % kTile, hq = threadIdx.x / kTile;
  float* out = a.scores + (int64_t)r * a.max_n;
  for (int t0 = blockIdx.y * kTile; t0 < n; t0 += gridDim.y * kTile) {
    __syncthreads();
    if (threadIdx.x < kTile) {
      const int i = t0 + threadIdx.x;
      prow_s[threadIdx.x] = i < n ? phys_row(a.bt, a.cache, seq, i, a.err) : -1;
    }
    __syncthreads();
    for (int x = threadIdx.x; x < kTile * Dk; x += blockDim.x) {
      const int te = x / Dk, d = x % Dk;
      const int64_t pr = prow_s[te];
      ks[te * ld + d] = pr >= 0 ? key_elem(a.cache, pr, d) : 0.f;
    }
    __syncthreads();
    float acc = 0.f;
    for (int h = hq; h < H; h += kQuarters) {
      const float* qh = qs + h * Dk;
      const float* ke = ks + e * ld;
      float dot = 0.f;
#pragma unroll 8
      for (int d = 0; d < Dk; ++d) dot = fmaf(qh[d], ke[d], dot);
      acc = fmaf(ws[h], fmaxf(dot, 0.f), acc);
    }
    part[hq * kTile + e] = acc;
    __syncthreads();
    if (threadIdx.x < kTile) {
      const int i = t0 + threadIdx.x;
      float s = 0.f;
#pragma unroll
      for (int q = 0; q < kQuarters; ++q) s += part[q * kTile + threadIdx.x];
      if (i < n) out[i] = prow_s[threadIdx.x] >= 0 ? s : -INFINITY;
    }
  }
}

}  // namespace

cudaError_t launch_indexer_scores(const IndexerArgs& a, int32_t n_rows, cudaStream_t s) {
  if (n_rows == 0 || a.max_n == 0) return cudaSuccess;
  const size_t smem = sizeof(float) * ((size_t)a.heads * a.dim + a.heads + (size_t)kTile * (a.dim + 1) +
                                       (size_t)kQuarters * kTile);
  cudaError_t e = cudaFuncSetAttribute(indexer_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const int tiles = (a.max_n + kTile - 1) / kTile;
  int gy = (2 * 152 * 2 + n_rows - 1) / n_rows;  // about four CTAs per SM in all
  if (gy > tiles) gy = tiles;
  if (gy < 1) gy = 1;
  return launch_k(indexer_scores_kernel, dim3(n_rows, gy), dim3(kThreads), smem, s, 0, a);
}

}  // namespace csa
