// Shared-K=V attention over selected compressed entries plus the raw sliding
// window, one joint softmax, inverse RoPE on the output, optional e4m3 output.
//
// Pages: "vLLM DeepSeek V4 Support", "DeepSeek V4 Attention Architecture"
// (shared key/value with inverse RoPE on the output, DSA top-k, a 128-token
// sliding window); "vLLM解密：DeepSeek-V4本地部署為何如此困難" §3.2 second
// fusion (inverse RoPE fused with the fp8 quantisation of the output).
//
// Generic CUDA-core kernel.  Grid (row, head group of 8, key split).  Each
// warp owns one query head; a tile of 32 keys is dequantised into shared
// memory, lane j scores key j, the warp updates its running max / sum and
// accumulates o += p_j * key_j with lane-strided dims.  With one split the
// epilogue normalises, applies the inverse rotation and stores; otherwise the
// split writes (m, l, o) and merge_kernel combines the splits.

#include "csa_kernels.h"

namespace csa {
namespace {

constexpr int kHeadsPerCta = 8;
constexpr int kThreads = 32 * kHeadsPerCta;
constexpr int kKeyTile = 32;
constexpr int kMaxDim = 512;

// Dequantised element d of physical row prow of cache c.
__device__ __forceinline__ float cache_elem(const csa_paged& c, int64_t prow, int d) {
  if (c.dtype == CSA_F32) return reinterpret_cast<const float*>(c.data)[prow * c.dim + d];
  if (c.dtype == CSA_BF16) return bf16_to_f32(reinterpret_cast<const uint16_t*>(c.data)[prow * c.dim + d]);
  const uint8_t* row = reinterpret_cast<const uint8_t*>(c.data) + prow * row_bytes(c);
  const int Dq = c.dtype == CSA_E4M3R ? c.dim - c.tail_bf16 : c.dim;
  if (d >= Dq) return bf16_to_f32(reinterpret_cast<const uint16_t*>(row + Dq)[d - Dq]);
  return e4m3_to_f32(row[d]) * reinterpret_cast<const float*>(c.scales)[prow];
}

// Inverse rotation of o (lane holds dims lane + 32*i) at position p, in place.
// Pair (d, d+1) lives in lanes (l, l^1) at the same i.
__device__ __forceinline__ void inverse_rope_lanes(float* o, int D, const RopeTab& rt, int64_t p) {
  const int lane = threadIdx.x & 31;
  const int R = rt.rope_dim;
#pragma unroll
  for (int i = 0; i < kMaxDim / 32; ++i) {
    const int d = lane + 32 * i;
    const float other = __shfl_xor_sync(0xffffffffu, o[i], 1);
    if (i < D / 32 && d >= D - R) {
      float c, s;
      rope_cs(rt, (d - (D - R)) / 2, p, c, s);
      // rotation by -angle: (x0, x1) -> (x0 c + x1 s, -x0 s + x1 c)
      o[i] = (d & 1) ? (-other * s + o[i] * c) : (o[i] * c + other * s);
    }
  }
}

__device__ void store_head(const AttnArgs& a, int r, int h, float* o) {
  const int lane = threadIdx.x & 31, D = a.dim;
  const int64_t base = ((int64_t)r * a.heads + h) * D;
  if (a.out_dtype == CSA_E4M3) {
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxDim / 32; ++i)
      if (i < D / 32) am = fmaxf(am, fabsf(o[i]));
    am = warp_max(am);
    const float inv = am > 0.f ? 448.0f / am : 0.0f;
    uint8_t* out = reinterpret_cast<uint8_t*>(a.out) + base;
#pragma unroll
    for (int i = 0; i < kMaxDim / 32; ++i)
      if (i < D / 32) out[lane + 32 * i] = f32_to_e4m3(o[i] * inv);
    if (lane == 0) a.out_scales[(int64_t)r * a.heads + h] = am / 448.0f;
  } else if (a.out_dtype == CSA_BF16) {
    uint16_t* out = reinterpret_cast<uint16_t*>(a.out) + base;
#pragma unroll
    for (int i = 0; i < kMaxDim / 32; ++i)
      if (i < D / 32) out[lane + 32 * i] = f32_to_bf16(o[i]);
  } else {
    float* out = reinterpret_cast<float*>(a.out) + base;
#pragma unroll
    for (int i = 0; i < kMaxDim / 32; ++i)
      if (i < D / 32) out[lane + 32 * i] = o[i];
  }
}

__global__ void __launch_bounds__(kThreads) attn_kernel(const AttnArgs a) {
  extern __shared__ float smem[];
  const int D = a.dim, ld = D + 1;
  float* qs = smem;                       // [8][D] rotated, pre-scaled queries
  float* ks = qs + kHeadsPerCta * D;      // [kKeyTile][D+1]
  __shared__ int64_t prow_s[kKeyTile];
  __shared__ int8_t which_s[kKeyTile];   // 0: comp, 1: swa, -1: masked

  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x, hg = blockIdx.y, split = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int h = hg * kHeadsPerCta + warp;
  const int seq = a.seq_id[r];
  const int64_t p = a.pos[r];
  const int32_t n_vis = n_visible((int32_t)p, a.ratio, a.window);
  const int32_t n_sel = a.topk ? a.k : n_vis;
  const int64_t w_lo = p - a.swa_len + 1 > 0 ? p - a.swa_len + 1 : 0;
  const int32_t n_win = (int32_t)(p - w_lo + 1);
  const int32_t n_keys = n_sel + n_win;
  const int32_t per = (n_keys + gridDim.z - 1) / gridDim.z;
  const int32_t j0 = split * per;
  const int32_t j1 = min(n_keys, j0 + per);

  // rotated query heads of this group, scaled by the softmax scale
  for (int x = threadIdx.x; x < kHeadsPerCta * D / 2; x += blockDim.x) {
    const int hh = x / (D / 2), d = 2 * (x % (D / 2));
    const int64_t qb = ((int64_t)r * a.heads + hg * kHeadsPerCta + hh) * D;
    float q0 = load_elem(a.q, a.q_dtype, qb + d), q1 = load_elem(a.q, a.q_dtype, qb + d + 1);
    if (d >= D - a.rope.rope_dim) {
      float c, s;
      rope_cs(a.rope, (d - (D - a.rope.rope_dim)) / 2, p, c, s);
      const float t0 = q0 * c - q1 * s;
      q1 = q0 * s + q1 * c;
      q0 = t0;
    }
    qs[hh * D + d] = q0 * a.scale;
    qs[hh * D + d + 1] = q1 * a.scale;
  }

  float o[kMaxDim / 32];
#pragma unroll
  for (int i = 0; i < kMaxDim / 32; ++i) o[i] = 0.f;
  float m = -INFINITY, l = 0.f;

  for (int t0 = j0; t0 < j1; t0 += kKeyTile) {
    __syncthreads();
    if (threadIdx.x < kKeyTile) {
      const int j = t0 + threadIdx.x;
      int64_t pr = -1;
      int8_t wh = -1;
      if (j < j1) {
        if (j < n_sel) {
          const int32_t idx = a.topk ? a.topk[(int64_t)r * a.k + j] : j;
          if (idx >= 0) {
            if (idx >= n_vis) {
              record_error(a.err, CSA_ERR_DEVICE_BOUNDS);
            } else {
              pr = phys_row(a.comp_bt, a.comp, seq, idx, a.err);
              wh = 0;
            }
          }
        } else {
          pr = phys_row(a.swa_bt, a.swa, seq, w_lo + (j - n_sel), a.err);
          wh = 1;
        }
      }
      prow_s[threadIdx.x] = pr;
      which_s[threadIdx.x] = pr >= 0 ? wh : (int8_t)-1;
    }
    __syncthreads();
    for (int x = threadIdx.x; x < kKeyTile * D; x += blockDim.x) {
      const int tj = x / D, d = x % D;
      const int8_t wh = which_s[tj];
      ks[tj * ld + d] = wh < 0 ? 0.f : cache_elem(wh == 0 ? a.comp : a.swa, prow_s[tj], d);
    }
    __syncthreads();
    // lane j scores key j for this warp's head
    const float* qh = qs + warp * D;
    const float* kj = ks + lane * ld;
    float logit = 0.f;
#pragma unroll 8
    for (int d = 0; d < D; ++d) logit = fmaf(qh[d], kj[d], logit);
    if (which_s[lane] < 0) logit = -INFINITY;
    const float tmax = warp_max(logit);
    const float m_new = fmaxf(m, tmax);
    if (m_new == -INFINITY) continue;  // whole tile masked, nothing seen yet
    const float pj = expf(logit - m_new);
    const float alpha = expf(m - m_new);
    l = l * alpha + warp_sum(pj);
    m = m_new;
#pragma unroll
    for (int i = 0; i < kMaxDim / 32; ++i) o[i] *= alpha;
    for (int j = 0; j < kKeyTile; ++j) {
      const float pb = __shfl_sync(0xffffffffu, pj, j);
      const float* kr = ks + j * ld;
#pragma unroll
      for (int i = 0; i < kMaxDim / 32; ++i)
        if (i < D / 32) o[i] = fmaf(pb, kr[lane + 32 * i], o[i]);
    }
  }

  if (gridDim.z == 1) {
    const float inv_l = l > 0.f ? 1.0f / l : 0.f;
#pragma unroll
    for (int i = 0; i < kMaxDim / 32; ++i) o[i] *= inv_l;
    inverse_rope_lanes(o, D, a.rope, p);
    store_head(a, r, h, o);
  } else {
    const int64_t pb = (((int64_t)r * a.heads + h) * gridDim.z + split);
    float* po = a.part_o + pb * D;
#pragma unroll
    for (int i = 0; i < kMaxDim / 32; ++i)
      if (i < D / 32) po[lane + 32 * i] = o[i];
    if (lane == 0) {
      a.part_ml[pb * 2] = m;
      a.part_ml[pb * 2 + 1] = l;
    }
  }
}

// One warp per (row, head): combine the splits' (m, l, o), normalise, rotate back, store.
__global__ void __launch_bounds__(32) merge_kernel(const AttnArgs a) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x, h = blockIdx.y, lane = threadIdx.x;
  const int S = a.n_splits, D = a.dim;
  const int64_t hb = ((int64_t)r * a.heads + h) * S;
  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, a.part_ml[(hb + s) * 2]);
  float o[kMaxDim / 32];
#pragma unroll
  for (int i = 0; i < kMaxDim / 32; ++i) o[i] = 0.f;
  float L = 0.f;
  for (int s = 0; s < S; ++s) {
    const float ms = a.part_ml[(hb + s) * 2];
    if (ms == -INFINITY) continue;
    const float f = expf(ms - M);
    L += a.part_ml[(hb + s) * 2 + 1] * f;
    const float* po = a.part_o + (hb + s) * D;
#pragma unroll
    for (int i = 0; i < kMaxDim / 32; ++i)
      if (i < D / 32) o[i] = fmaf(po[lane + 32 * i], f, o[i]);
  }
  const float inv_l = L > 0.f ? 1.0f / L : 0.f;
#pragma unroll
  for (int i = 0; i < kMaxDim / 32; ++i) o[i] *= inv_l;
  inverse_rope_lanes(o, D, a.rope, a.pos[r]);
  store_head(a, r, h, o);
}

}  // namespace

int32_t attn_splits(int32_t n_rows, int32_t heads, int32_t keys_per_row) {
  const int64_t ctas = (int64_t)n_rows * (heads / kHeadsPerCta);
  const int64_t target = 152 * 4;
  int64_t s = (target + ctas - 1) / ctas;
  const int64_t max_s = (keys_per_row + 63) / 64;  // at least ~64 keys per split
  if (s > max_s) s = max_s;
  if (s < 1) s = 1;
  if (s > 64) s = 64;
  return (int32_t)s;
}

size_t attn_workspace_bytes(int32_t n_rows, int32_t heads, int32_t dim, int32_t n_splits) {
  if (n_splits <= 1) return 0;
  return sizeof(float) * (size_t)n_rows * heads * n_splits * (dim + 2);
}

cudaError_t launch_attn(const AttnArgs& a, int32_t n_rows, int32_t keys_per_row, cudaStream_t s) {
  (void)keys_per_row;
  if (n_rows == 0) return cudaSuccess;
  const size_t smem = sizeof(float) * ((size_t)kHeadsPerCta * a.dim + (size_t)kKeyTile * (a.dim + 1));
  cudaError_t e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_k(attn_kernel, dim3(n_rows, a.heads / kHeadsPerCta, a.n_splits), dim3(kThreads), smem, s, 0,
               a);
  if (e != cudaSuccess || a.n_splits == 1) return e;
  return launch_attn_merge(a, n_rows, s);
}

cudaError_t launch_attn_merge(const AttnArgs& a, int32_t n_rows, cudaStream_t s) {
  return launch_k(merge_kernel, dim3(n_rows, a.heads), dim3(32), 0, s, 0, a);
}

}  // namespace csa
