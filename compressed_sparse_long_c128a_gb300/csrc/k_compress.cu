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

// Threads of the key path: warps 0-7.  With the query norm fused in
// (csa_compress_insert_qnorm), warps 8-15 of the same CTA normalise the
// token's query heads meanwhile (static dispatch by warp ID), so the key path
// synchronises on named barrier 1 over its own 256 threads only.
constexpr int kThreads = 256;
constexpr int kQThreads = 256;  // query-norm warps

__device__ __forceinline__ void grp_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }

// Sum / max over the key path's 256 threads; `red` is shared scratch of >= 8 floats.
__device__ __forceinline__ float group_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  v = warp_sum(v);
  grp_sync();
  if (lane == 0) red[wid] = v;
  grp_sync();
  return warp_sum(lane < kThreads / 32 ? red[lane] : 0.f);
}
__device__ __forceinline__ float group_max(float v, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  v = warp_max(v);
  grp_sync();
  if (lane == 0) red[wid] = v;
  grp_sync();
  return warp_max(lane < kThreads / 32 ? red[lane] : 0.f);
}

__device__ __forceinline__ void store_elem(void* base, int32_t dtype, int64_t idx, float v) {
  if (dtype == CSA_F32)
    reinterpret_cast<float*>(base)[idx] = v;
  else
    reinterpret_cast<uint16_t*>(base)[idx] = f32_to_bf16(v);
}

// Write y[0..D) (shared memory) as physical row `prow` of cache c.  Called by
// the whole block with a block-uniform prow >= 0.
__device__ void store_row(const csa_paged& c, int64_t prow, const float* y, int D, float* red) {
  if (c.dtype == CSA_E4M3R) {  // e4m3 + per-row scale over [0, D - tail), bf16 tail
    const int Dq = D - c.tail_bf16;
    float am = 0.f;
    for (int d = threadIdx.x; d < Dq; d += kThreads) am = fmaxf(am, fabsf(y[d]));
    am = group_max(am, red);
    const float inv = am > 0.f ? 448.0f / am : 0.0f;
    uint8_t* row = reinterpret_cast<uint8_t*>(c.data) + prow * row_bytes(c);
    for (int pr = threadIdx.x; pr < Dq / 2; pr += kThreads)
      *reinterpret_cast<uint16_t*>(row + 2 * pr) = f32x2_to_e4m3x2(y[2 * pr] * inv, y[2 * pr + 1] * inv);
    for (int pr = threadIdx.x; pr < c.tail_bf16 / 2; pr += kThreads)
      *reinterpret_cast<uint32_t*>(row + Dq + 4 * pr) = f32x2_to_bf16x2(y[Dq + 2 * pr], y[Dq + 2 * pr + 1]);
    if (threadIdx.x == 0) reinterpret_cast<float*>(c.scales)[prow] = am / 448.0f;
  } else if (c.dtype == CSA_E4M3) {
    float am = 0.f;
    for (int d = threadIdx.x; d < D; d += kThreads) am = fmaxf(am, fabsf(y[d]));
    am = group_max(am, red);
    const float scale = am / 448.0f;
    const float inv = am > 0.f ? 448.0f / am : 0.0f;
    uint8_t* row = reinterpret_cast<uint8_t*>(c.data) + prow * (int64_t)D;
    for (int pr = threadIdx.x; pr < D / 2; pr += kThreads)
      *reinterpret_cast<uint16_t*>(row + 2 * pr) = f32x2_to_e4m3x2(y[2 * pr] * inv, y[2 * pr + 1] * inv);
    if (threadIdx.x == 0) reinterpret_cast<float*>(c.scales)[prow] = scale;
  } else if (c.dtype == CSA_E2M1) {  // one thread per group of 16 (D % 16 == 0)
    uint8_t* row = reinterpret_cast<uint8_t*>(c.data) + prow * (int64_t)(D / 2);
    uint8_t* srow = reinterpret_cast<uint8_t*>(c.scales) + prow * (int64_t)(D / 16);
    for (int g = threadIdx.x; g < D / 16; g += kThreads) {
      uint2 packed;
      srow[g] = quantize_e2m1_group(y + 16 * g, packed);
      *reinterpret_cast<uint2*>(row + g * 8) = packed;
    }
  } else if (c.dtype == CSA_BF16) {
    uint16_t* row = reinterpret_cast<uint16_t*>(c.data) + prow * (int64_t)D;
    for (int pr = threadIdx.x; pr < D / 2; pr += kThreads) {
      uint32_t v = (uint32_t)f32_to_bf16(y[2 * pr]) | ((uint32_t)f32_to_bf16(y[2 * pr + 1]) << 16);
      *reinterpret_cast<uint32_t*>(row + 2 * pr) = v;
    }
  } else {
    float* row = reinterpret_cast<float*>(c.data) + prow * (int64_t)D;
    for (int pr = threadIdx.x; pr < D / 2; pr += kThreads)
      *reinterpret_cast<float2*>(row + 2 * pr) = make_float2(y[2 * pr], y[2 * pr + 1]);
  }
}

// y := RoPE(y * inv_rms * gamma, pos) in place, pairs (2k, 2k+1) over the last r dims.
__device__ void norm_rope_inplace(float* y, int D, float inv_rms, const float* gamma, const RopeTab& rt,
                                  int64_t pos) {
  const int R = rt.rope_dim;
  for (int pr = threadIdx.x; pr < D / 2; pr += kThreads) {
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

// Eight consecutive elements of a row in `dtype` (F32 or BF16) as floats; 16-byte (bf16) or
// 2 x 16-byte (f32) loads, so `p` must be 16-byte aligned.
__device__ __forceinline__ void load8(const void* base, int32_t dtype, int64_t idx, float* v) {
  if (dtype == CSA_F32) {
    const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + idx);
    const float4 a = p[0], b = p[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(base) + idx);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[2 * e] = bf16_to_f32((uint16_t)(w[e] & 0xFFFF));
      v[2 * e + 1] = bf16_to_f32((uint16_t)(w[e] >> 16));
    }
  }
}

__device__ __forceinline__ void store8(void* base, int32_t dtype, int64_t idx, const float* v) {
  if (dtype == CSA_F32) {
    float4* p = reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + idx);
    p[0] = make_float4(v[0], v[1], v[2], v[3]);
    p[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else {
    *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(base) + idx) =
        make_uint4(f32x2_to_bf16x2(v[0], v[1]), f32x2_to_bf16x2(v[2], v[3]), f32x2_to_bf16x2(v[4], v[5]),
                   f32x2_to_bf16x2(v[6], v[7]));
  }
}

// Warps 8-15 of a CTA with the query norm fused in: the RMSNorm of each head of
// query row j (the row of token j), RoPE left to the attention kernel.  Lane l
// holds elements [8l, 8l+8) and [256+8l, 256+8l+8) of a head (D <= 512).
__device__ void qnorm_role(const QNormArgs& q, int64_t j, int qt) {
  const int lane = qt & 31, w = qt >> 5;
  const int D = q.dim;
  for (int h = w; h < q.heads; h += kQThreads / 32) {
    const int64_t base = (j * q.heads + h) * D;
    float x[2][8];
    float ss = 0.f;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int d0 = 8 * lane + 256 * u;
      if (d0 < D) {
        load8(q.q, q.q_dtype, base + d0, x[u]);
#pragma unroll
        for (int e = 0; e < 8; ++e) ss += x[u][e] * x[u][e];
      }
    }
    ss = warp_sum(ss);
    const float inv = 1.0f / sqrtf(ss / (float)D + q.eps);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int d0 = 8 * lane + 256 * u;
      if (d0 < D) {
        const float4* g4 = reinterpret_cast<const float4*>(q.gamma + d0);
        const float4 g0 = g4[0], g1 = g4[1];
        const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = x[u][e] * inv * g[e];
        store8(q.out, q.out_dtype, base + d0, y);
      }
    }
  }
}

template <bool kQ>
__global__ void __launch_bounds__(kQ ? kThreads + kQThreads : kThreads) ingest_kernel(const IngestArgs a,
                                                                                     const QNormArgs qa) {
  extern __shared__ float y[];
  __shared__ float red[32];
  pdl_trigger();
  pdl_wait();
  if constexpr (kQ) {
    if (threadIdx.x >= kThreads) {  // warps 8-15: the query norm
      qnorm_role(qa, blockIdx.x, threadIdx.x - kThreads);
      return;
    }
  }
  const int j = blockIdx.x;
  const int D = a.dim;
  const int seq = a.seq_id[j];
  const int64_t p = a.pos[j];
  const int64_t srow = phys_row(a.state_bt, a.state, seq, p, a.err);
  const int64_t wrow = a.swa.data ? phys_row(a.swa_bt, a.swa, seq, p, a.err) : -1;  // no window cache: state only

  float ss = 0.f;
  for (int d = threadIdx.x; d < D; d += kThreads) {
    float x = load_elem(a.kv, a.in_dtype, (int64_t)j * D + d);
    y[d] = x;
    ss += x * x;
    if (srow >= 0) {
      float g = load_elem(a.gate, a.in_dtype, (int64_t)j * D + d);
      store_elem(a.state.data, a.state.dtype, srow * 2 * D + d, x);
      store_elem(a.state.data, a.state.dtype, srow * 2 * D + D + d, g);
    }
  }
  ss = group_sum(ss, red);
  if (wrow < 0) return;  // block-uniform
  const float inv = 1.0f / sqrtf(ss / (float)D + a.eps);
  grp_sync();
  norm_rope_inplace(y, D, inv, a.gamma_swa, a.rope, p);
  grp_sync();
  store_row(a.swa, wrow, y, D, red);
}

__global__ void __launch_bounds__(kThreads) emit_kernel(const EmitArgs a) {
  extern __shared__ float y[];
  __shared__ float red[32];
  __shared__ int64_t rows[256];
  __shared__ int bad;
  pdl_trigger();
  // every CTA waits, even one with nothing to emit: this grid may only complete
  // after the ingest launch has, so later launches that wait on this one also
  // see ingest's writes
  pdl_wait();
  const int j = blockIdx.x;
  const int64_t t = a.pos[j];
  const int W = a.window, Rt = a.ratio, D = a.dim;
  if (t < W - 1 || (t - W + 1) % Rt) return;  // no window closes at this token
  const int64_t i = (t - W + 1) / Rt;
  const int64_t base = i * Rt;  // first raw position = anchor
  const int seq = a.seq_id[j];

  if (threadIdx.x == 0) bad = 0;
  grp_sync();
  for (int o = threadIdx.x; o < W; o += kThreads) {
    int64_t r = phys_row(a.state_bt, a.state, seq, base + o, a.err);
    rows[o] = r;
    if (r < 0) bad = 1;
  }
  const int64_t crow = phys_row(a.comp_bt, a.comp, seq, i, a.err);
  grp_sync();
  if (bad || crow < 0) return;

  const int sdt = a.state.dtype;
  float ss = 0.f;
  for (int pr = threadIdx.x; pr < D / 2; pr += kThreads) {
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
  ss = group_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / (float)D + a.eps);
  grp_sync();
  norm_rope_inplace(y, D, inv, a.gamma_c, a.rope, base);
  grp_sync();
  store_row(a.comp, crow, y, D, red);
}

// ------------------------------------------------------------------ one launch for decode-sized calls

constexpr int kFusedMaxTokens = 1024;  // the (seq, pos) scan of an emitting CTA stays cheap
constexpr int kFusedMaxDim = 512;
constexpr int kQuarters = 4;  // window rows split over four groups of threads per 8-channel group

// CTA j takes token j of the call: state row and window row as ingest_kernel
// writes them; then, if a window closes at the token, the entry as emit_kernel
// forms it, but with every window row that is one of the call's own tokens
// read from the call's inputs (the state cache holds the rest, written by
// earlier calls), so no CTA depends on another CTA's writes.
template <bool kQ>
__global__ void __launch_bounds__(kQ ? kThreads + kQThreads : kThreads)
    compress_fused_kernel(const IngestArgs ia, const EmitArgs ea, int32_t n_tok, const QNormArgs qa) {
  __shared__ float y[kFusedMaxDim];
  __shared__ float red[32];
  __shared__ float part[kQuarters][3][kFusedMaxDim];  // per row group: running max, denominator, weighted sum
  __shared__ const void* src_kv[256];                  // window row o: kv and gate of the row
  __shared__ const void* src_gate[256];
  __shared__ int32_t src_dt[256];
  __shared__ int in_call[256];
  __shared__ int bad;
  pdl_trigger();
  pdl_wait();
  if constexpr (kQ) {
    if (threadIdx.x >= kThreads) {  // warps 8-15: the query norm
      qnorm_role(qa, blockIdx.x, threadIdx.x - kThreads);
      return;
    }
  }
  const int j = blockIdx.x;
  const int D = ia.dim, G8 = D / 8;
  // every load that depends only on j first: the token's raw row with its
  // position (one memory latency), then all block-table lookups of the CTA
  // (a second), then the ingest's writes; the window rows of the emission
  // are the third and last dependent read
  float x[8], gt[8];
  const bool has_g = threadIdx.x < G8;  // D <= 512: one 8-channel group per thread
  if (has_g) {
    load8(ia.kv, ia.in_dtype, (int64_t)j * D + 8 * threadIdx.x, x);
    load8(ia.gate, ia.in_dtype, (int64_t)j * D + 8 * threadIdx.x, gt);
  }
  const int seq = ia.seq_id[j];
  const int64_t p = ia.pos[j];
  const int W = ea.window, Rt = ea.ratio;
  const bool emits = p >= W - 1 && (p - W + 1) % Rt == 0;  // block-uniform
  const int64_t i = emits ? (p - W + 1) / Rt : 0;
  const int64_t base = i * Rt;
  const int64_t srow = phys_row(ia.state_bt, ia.state, seq, p, ia.err);
  const int64_t wrow = ia.swa.data ? phys_row(ia.swa_bt, ia.swa, seq, p, ia.err) : -1;
  int64_t crow = -1;
  if (emits) {
    crow = phys_row(ea.comp_bt, ea.comp, seq, i, ea.err);
    // window row o from the state cache unless it is one of the call's tokens
    // (those are read from the inputs: another CTA writes their state rows)
    for (int o = threadIdx.x; o < W; o += kThreads) {
      in_call[o] = -1;
      const int64_t r = phys_row(ea.state_bt, ea.state, seq, base + o, ea.err);
      const size_t eb = ea.state.dtype == CSA_F32 ? 4 : 2;
      src_kv[o] = r < 0 ? nullptr : reinterpret_cast<const uint8_t*>(ea.state.data) + r * 2 * D * eb;
      src_gate[o] = r < 0 ? nullptr : reinterpret_cast<const uint8_t*>(ea.state.data) + (r * 2 * D + D) * eb;
      src_dt[o] = ea.state.dtype;
    }
    grp_sync();
    for (int k = threadIdx.x; k < n_tok; k += kThreads) {
      const int64_t q = ea.pos[k];
      if (ea.seq_id[k] == seq && q >= base && q < base + W) in_call[q - base] = k;
    }
  }

  // ---- ingest
  float ss = 0.f;
  if (has_g) {
    if (srow >= 0) {
      store8(ia.state.data, ia.state.dtype, srow * 2 * D + 8 * threadIdx.x, x);
      store8(ia.state.data, ia.state.dtype, srow * 2 * D + D + 8 * threadIdx.x, gt);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      y[8 * threadIdx.x + e] = x[e];
      ss += x[e] * x[e];
    }
  }
  ss = group_sum(ss, red);
  if (wrow >= 0) {  // block-uniform
    const float inv = 1.0f / sqrtf(ss / (float)D + ia.eps);
    grp_sync();
    norm_rope_inplace(y, D, inv, ia.gamma_swa, ia.rope, p);
    grp_sync();
    store_row(ia.swa, wrow, y, D, red);
  }

  // ---- emission of the entry whose window closes at this token
  if (!emits) return;
  grp_sync();  // y and red are reused below; in_call is complete
  if (threadIdx.x == 0) bad = 0;
  grp_sync();
  for (int o = threadIdx.x; o < W; o += kThreads) {
    const int k = in_call[o];
    if (k >= 0) {
      src_kv[o] = reinterpret_cast<const uint8_t*>(ia.kv) + (int64_t)k * D * (ia.in_dtype == CSA_F32 ? 4 : 2);
      src_gate[o] = reinterpret_cast<const uint8_t*>(ia.gate) + (int64_t)k * D * (ia.in_dtype == CSA_F32 ? 4 : 2);
      src_dt[o] = ia.in_dtype;
    } else if (!src_kv[o]) {
      bad = 1;
    }
  }
  grp_sync();
  if (bad || crow < 0) return;

  // online softmax over the window offsets, per channel: thread (g, qtr) takes
  // channels [8g, 8g+8) and offsets qtr, qtr+4, ...; the four row groups merge below
  for (int x = threadIdx.x; x < G8 * kQuarters; x += kThreads) {
    const int g = x % G8, qtr = x / G8;
    float m[8], sm[8], c[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      m[e] = -INFINITY;
      sm[e] = 0.f;
      c[e] = 0.f;
    }
    for (int o = qtr; o < W; o += kQuarters) {
      float kv[8], gt[8];
      load8(src_kv[o], src_dt[o], 8 * g, kv);
      load8(src_gate[o], src_dt[o], 8 * g, gt);
      const float4* b4 = reinterpret_cast<const float4*>(ea.bias + (int64_t)o * D + 8 * g);
      const float4 b0 = b4[0], b1 = b4[1];
      const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float z = gt[e] + bb[e];
        if (z > m[e]) {
          const float f = expf(m[e] - z);
          sm[e] = sm[e] * f + 1.f;
          c[e] = c[e] * f + kv[e];
          m[e] = z;
        } else {
          const float ez = expf(z - m[e]);
          sm[e] += ez;
          c[e] += ez * kv[e];
        }
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      part[qtr][0][8 * g + e] = m[e];
      part[qtr][1][8 * g + e] = sm[e];
      part[qtr][2][8 * g + e] = c[e];
    }
  }
  grp_sync();
  float ss2 = 0.f;
  for (int d = threadIdx.x; d < D; d += kThreads) {
    float mx = -INFINITY;
#pragma unroll
    for (int q = 0; q < kQuarters; ++q) mx = fmaxf(mx, part[q][0][d]);
    float sm = 0.f, c = 0.f;
#pragma unroll
    for (int q = 0; q < kQuarters; ++q) {
      const float mq = part[q][0][d];
      if (mq == -INFINITY) continue;  // a row group with no offsets (W < 4)
      const float f = expf(mq - mx);
      sm += part[q][1][d] * f;
      c += part[q][2][d] * f;
    }
    const float v = c / sm;
    y[d] = v;
    ss2 += v * v;
  }
  ss2 = group_sum(ss2, red);
  const float inv = 1.0f / sqrtf(ss2 / (float)D + ea.eps);
  grp_sync();
  norm_rope_inplace(y, D, inv, ea.gamma_c, ea.rope, base);
  grp_sync();
  store_row(ea.comp, crow, y, D, red);
}

}  // namespace

bool compress_fused_eligible(const IngestArgs& ia, const EmitArgs& ea, int32_t n_tok) {
  const uintptr_t al = reinterpret_cast<uintptr_t>(ia.kv) | reinterpret_cast<uintptr_t>(ia.gate) |
                       reinterpret_cast<uintptr_t>(ia.state.data) | reinterpret_cast<uintptr_t>(ea.bias);
  return n_tok <= kFusedMaxTokens && ia.dim % 8 == 0 && ia.dim <= kFusedMaxDim && ea.window <= 256 && al % 16 == 0;
}

cudaError_t launch_compress_fused(const IngestArgs& ia, const EmitArgs& ea, const QNormArgs& q, int32_t n_tok,
                                  cudaStream_t s) {
  if (n_tok == 0) return cudaSuccess;
  if (q.q) return launch_k(compress_fused_kernel<true>, dim3(n_tok), dim3(kThreads + kQThreads), 0, s, 0, ia, ea, n_tok, q);
  return launch_k(compress_fused_kernel<false>, dim3(n_tok), dim3(kThreads), 0, s, 0, ia, ea, n_tok, q);
}

cudaError_t launch_ingest(const IngestArgs& a, const QNormArgs& q, int32_t n_tok, cudaStream_t s) {
  if (n_tok == 0) return cudaSuccess;
  const size_t smem = a.dim * sizeof(float);
  if (q.q) return launch_k(ingest_kernel<true>, dim3(n_tok), dim3(kThreads + kQThreads), smem, s, 0, a, q);
  return launch_k(ingest_kernel<false>, dim3(n_tok), dim3(kThreads), smem, s, 0, a, q);
}

cudaError_t launch_emit(const EmitArgs& a, int32_t n_tok, cudaStream_t s) {
  if (n_tok == 0) return cudaSuccess;
  return launch_k(emit_kernel, dim3(n_tok), dim3(kThreads), a.dim * sizeof(float), s, 0, a);
}

}  // namespace csa
