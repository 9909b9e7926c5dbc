// HBM-bound kernels of the training step: RMSNorm forward/backward (with the
// residual add and deterministic gain-gradient reduction), per-head QK
// RMSNorm + RoPE-neox forward/backward, the cross-entropy finalise and
// softmax-gradient passes, the multi-buffer squared sum, the clip scale and
// AdamW. All are single-pass (or two-pass where a row statistic is needed),
// 128-bit vectorised, with warp-shuffle reductions; every reduction runs in a
// fixed order, so results are bitwise reproducible run to run.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace rdt {

// ----------------------------------------------------------------- RMSNorm
// One warp per row; lane j-th float4 chunk is column 4*(lane + 32*j).
template <int NJ>
__global__ void __launch_bounds__(256) rmsnorm_fwd_kernel(const float* __restrict__ x,
                                                          const float* __restrict__ gamma,
                                                          bf16* __restrict__ y,
                                                          float* __restrict__ rstd, int T, int H,
                                                          float eps) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= T) return;
  const int H4 = H >> 2;
  const float4* xr = reinterpret_cast<const float4*>(x + (int64_t)row * H);
  float4 v[NJ];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int c = lane + 32 * j;
    if (c < H4) {
      v[j] = xr[c];
      ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
    }
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / H + eps);
  const float4* g4 = reinterpret_cast<const float4*>(gamma);
  uint2* yr = reinterpret_cast<uint2*>(y + (int64_t)row * H);
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int c = lane + 32 * j;
    if (c < H4) {
      const float4 g = g4[c];
      uint2 o;
      o.x = pack_bf16x2(v[j].x * r * g.x, v[j].y * r * g.y);
      o.y = pack_bf16x2(v[j].z * r * g.z, v[j].w * r * g.w);
      yr[c] = o;
    }
  }
  if (lane == 0) rstd[row] = r;
}

// dx = r*(dy*g - xhat*mean(dy*g*xhat)) + resid; per-CTA partial of sum(dy*xhat).
template <int NJ>
__global__ void __launch_bounds__(256) rmsnorm_bwd_kernel(
    const float* __restrict__ dy, const float* __restrict__ x, const float* __restrict__ rstd,
    const float* __restrict__ gamma, const float* __restrict__ resid, float* __restrict__ dx,
    bf16* __restrict__ dxb, float* __restrict__ partials, int T, int H) {
  extern __shared__ float red[];  // [H]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H4 = H >> 2;
  const float4* g4 = reinterpret_cast<const float4*>(gamma);
  float4 acc[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);

  for (int row = blockIdx.x * 8 + warp; row < T; row += gridDim.x * 8) {
    const float4* dyr = reinterpret_cast<const float4*>(dy + (int64_t)row * H);
    const float4* xr = reinterpret_cast<const float4*>(x + (int64_t)row * H);
    const float r = rstd[row];
    float dot = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int c = lane + 32 * j;
      if (c < H4) {
        const float4 a = dyr[c], b = xr[c], g = g4[c];
        dot += a.x * g.x * b.x + a.y * g.y * b.y + a.z * g.z * b.z + a.w * g.w * b.w;
      }
    }
    dot = warp_sum(dot) * r;  // sum(dy*g*xhat)
    const float cmean = dot / H;
    float4* dxr = reinterpret_cast<float4*>(dx + (int64_t)row * H);
    const float4* rr = resid ? reinterpret_cast<const float4*>(resid + (int64_t)row * H) : nullptr;
    uint2* dbr = dxb ? reinterpret_cast<uint2*>(dxb + (int64_t)row * H) : nullptr;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int c = lane + 32 * j;
      if (c < H4) {
        const float4 a = dyr[c], b = xr[c], g = g4[c];
        const float4 xh = make_float4(b.x * r, b.y * r, b.z * r, b.w * r);
        float4 o = make_float4(r * (a.x * g.x - xh.x * cmean), r * (a.y * g.y - xh.y * cmean),
                               r * (a.z * g.z - xh.z * cmean), r * (a.w * g.w - xh.w * cmean));
        if (rr) {
          const float4 q = rr[c];
          o.x += q.x; o.y += q.y; o.z += q.z; o.w += q.w;
        }
        dxr[c] = o;
        if (dbr) {
          uint2 ob;
          ob.x = pack_bf16x2(o.x, o.y);
          ob.y = pack_bf16x2(o.z, o.w);
          dbr[c] = ob;
        }
        acc[j].x += a.x * xh.x;
        acc[j].y += a.y * xh.y;
        acc[j].z += a.z * xh.z;
        acc[j].w += a.w * xh.w;
      }
    }
  }
  // fixed-order reduction of the 8 warps' gain partials
  for (int w = 0; w < 8; ++w) {
    if (warp == w) {
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const int c = lane + 32 * j;
        if (c < H4) {
          float4* s4 = reinterpret_cast<float4*>(red) + c;
          if (w == 0) {
            *s4 = acc[j];
          } else {
            float4 t = *s4;
            t.x += acc[j].x; t.y += acc[j].y; t.z += acc[j].z; t.w += acc[j].w;
            *s4 = t;
          }
        }
      }
    }
    __syncthreads();
  }
  for (int c = threadIdx.x; c < H; c += blockDim.x) partials[(int64_t)blockIdx.x * H + c] = red[c];
}

// out[c] = sum_p partials[p, c] in order p = 0, 1, ...
__global__ void reduce_cols_kernel(const float* __restrict__ partials, int P, int W,
                                   float* __restrict__ out) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= W) return;
  float s = 0.f;
  for (int p = 0; p < P; ++p) s += partials[(int64_t)p * W + c];
  out[c] = s;
}

#define RDT_NJ_SWITCH(KERNEL, H, GRID, BLOCK, SMEM, STREAM, ...)                           \
  do {                                                                                     \
    note_launch();                                                                         \
    const int nj_need = ((H) / 4 + 31) / 32;                                               \
    if (nj_need <= 1) KERNEL<1><<<GRID, BLOCK, SMEM, STREAM>>>(__VA_ARGS__);               \
    else if (nj_need <= 2) KERNEL<2><<<GRID, BLOCK, SMEM, STREAM>>>(__VA_ARGS__);          \
    else if (nj_need <= 4) KERNEL<4><<<GRID, BLOCK, SMEM, STREAM>>>(__VA_ARGS__);          \
    else if (nj_need <= 8) KERNEL<8><<<GRID, BLOCK, SMEM, STREAM>>>(__VA_ARGS__);          \
    else if (nj_need <= 12) KERNEL<12><<<GRID, BLOCK, SMEM, STREAM>>>(__VA_ARGS__);        \
    else if (nj_need <= 16) KERNEL<16><<<GRID, BLOCK, SMEM, STREAM>>>(__VA_ARGS__);        \
    else if (nj_need <= 20) KERNEL<20><<<GRID, BLOCK, SMEM, STREAM>>>(__VA_ARGS__);        \
    else if (nj_need <= 24) KERNEL<24><<<GRID, BLOCK, SMEM, STREAM>>>(__VA_ARGS__);        \
    else KERNEL<32><<<GRID, BLOCK, SMEM, STREAM>>>(__VA_ARGS__);                           \
  } while (0)

cudaError_t rmsnorm_fwd(const float* x, const float* gamma, bf16* y, float* rstd, int T, int H,
                        float eps, cudaStream_t s) {
  const dim3 grid((T + 7) / 8);
  RDT_NJ_SWITCH(rmsnorm_fwd_kernel, H, grid, 256, 0, s, x, gamma, y, rstd, T, H, eps);
  return cudaGetLastError();
}

int rmsnorm_bwd_partial_rows(int T) {
  const int want = (T + 7) / 8;
  const int cap = min(2 * num_sms(), kMaxPartialRows);
  return want < cap ? want : cap;
}

cudaError_t rmsnorm_bwd(const float* dy, const float* x, const float* rstd, const float* gamma,
                        const float* resid, float* dx, bf16* dx_bf16, float* dgamma,
                        float* partials, int T, int H, cudaStream_t s) {
  const int P = rmsnorm_bwd_partial_rows(T);
  RDT_NJ_SWITCH(rmsnorm_bwd_kernel, H, dim3(P), 256, H * sizeof(float), s, dy, x, rstd, gamma,
                resid, dx, dx_bf16, partials, T, H);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  note_launch();
  reduce_cols_kernel<<<(H + 255) / 256, 256, 0, s>>>(partials, P, H, dgamma);
  return cudaGetLastError();
}

// ----------------------------------------------------------------- RoPE table
// cs[s, i] = (cos, sin)(s * theta^(-2i/d)), evaluated in fp64, stored fp32.
__global__ void rope_table_kernel(float2* __restrict__ cs, int S, int d, double theta) {
  const int half = d / 2;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= S * half) return;
  const int s = idx / half, i = idx % half;
  const double inv = pow(theta, -2.0 * i / d);
  double sn, cn;
  sincos(static_cast<double>(s) * inv, &sn, &cn);
  cs[idx] = make_float2(static_cast<float>(cn), static_cast<float>(sn));
}

cudaError_t rope_table(float* cs, int S, int d, float theta, cudaStream_t s) {
  const int n = S * (d / 2);
  note_launch();
  rope_table_kernel<<<(n + 255) / 256, 256, 0, s>>>(reinterpret_cast<float2*>(cs), S, d,
                                                    static_cast<double>(theta));
  return cudaGetLastError();
}

// ----------------------------------------------------- QK RMSNorm + RoPE fwd
// One warp per (token, head) over nh query heads then nkv key heads. Lane l
// owns the rotation pairs (2l + 64j, 2l + 1 + 64j) and their partners + d/2.
__global__ void __launch_bounds__(256) qknorm_rope_fwd_kernel(
    const bf16* __restrict__ qkv, int64_t ld, bf16* __restrict__ qo, bf16* __restrict__ ko,
    float* __restrict__ rq, float* __restrict__ rk, const float* __restrict__ gq,
    const float* __restrict__ gk, const float2* __restrict__ cs, int T, int S, int nh, int nkv,
    int d, float eps) {
  const int64_t item = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int heads = nh + nkv;
  if (item >= (int64_t)T * heads) return;
  const int t = static_cast<int>(item / heads), hd = static_cast<int>(item % heads);
  const bool isq = hd < nh;
  const int h = isq ? hd : hd - nh;
  const bf16* src = qkv + (int64_t)t * ld + (isq ? h * d : nh * d + h * d);
  bf16* dst = isq ? qo + (int64_t)t * nh * d + h * d : ko + (int64_t)t * nkv * d + h * d;
  const float* g = isq ? gq : gk;
  const int half = d / 2, pos = t % S;
  float x0[2][2], x1[2][2];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int i = 2 * lane + 64 * j;
    if (i < half) {
      const uint32_t a = *reinterpret_cast<const uint32_t*>(src + i);
      const uint32_t b = *reinterpret_cast<const uint32_t*>(src + half + i);
      x0[j][0] = bf16lo(a); x0[j][1] = bf16hi(a);
      x1[j][0] = bf16lo(b); x1[j][1] = bf16hi(b);
      ss += x0[j][0] * x0[j][0] + x0[j][1] * x0[j][1] + x1[j][0] * x1[j][0] + x1[j][1] * x1[j][1];
    }
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / d + eps);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int i = 2 * lane + 64 * j;
    if (i < half) {
      float o0[2], o1[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float y0 = x0[j][e] * r * g[i + e];
        const float y1 = x1[j][e] * r * g[half + i + e];
        const float2 c = cs[(int64_t)pos * half + i + e];
        o0[e] = y0 * c.x - y1 * c.y;
        o1[e] = y1 * c.x + y0 * c.y;
      }
      *reinterpret_cast<uint32_t*>(dst + i) = pack_bf16x2(o0[0], o0[1]);
      *reinterpret_cast<uint32_t*>(dst + half + i) = pack_bf16x2(o1[0], o1[1]);
    }
  }
  if (lane == 0) {
    if (isq) rq[(int64_t)t * nh + h] = r;
    else rk[(int64_t)t * nkv + h] = r;
  }
}

cudaError_t qknorm_rope_fwd(const bf16* qkv, int64_t ld_qkv, bf16* q_out, bf16* k_out,
                            float* rstd_q, float* rstd_k, const float* gq, const float* gk,
                            const float* cs, int T, int S, int nh, int nkv, int d, float eps,
                            cudaStream_t s) {
  const int64_t items = (int64_t)T * (nh + nkv);
  note_launch();
  qknorm_rope_fwd_kernel<<<(unsigned)((items + 7) / 8), 256, 0, s>>>(
      qkv, ld_qkv, q_out, k_out, rstd_q, rstd_k, gq, gk, reinterpret_cast<const float2*>(cs), T, S,
      nh, nkv, d, eps);
  return cudaGetLastError();
}

// ----------------------------------------------------- QK RMSNorm + RoPE bwd
// Inverse rotation of the incoming gradient, then the RMSNorm backward over
// head_dim. Gain gradients: per-lane register partials, fixed-order CTA
// reduction into partials[block, 2*d] (q gains then k gains).
__global__ void __launch_bounds__(256) qknorm_rope_bwd_kernel(
    const float* __restrict__ dq, const float* __restrict__ dk, const bf16* __restrict__ qkv,
    int64_t ld, const float* __restrict__ rq, const float* __restrict__ rk,
    const float* __restrict__ gq, const float* __restrict__ gk, const float2* __restrict__ cs,
    bf16* __restrict__ dqkv, float* __restrict__ partials, int T, int S, int nh, int nkv, int d) {
  __shared__ float red[8][2][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int heads = nh + nkv;
  const int half = d / 2;
  float accq[2][2][2] = {}, acck[2][2][2] = {};  // [j][half][e]
  const int64_t items = (int64_t)T * heads;
  for (int64_t item = (int64_t)blockIdx.x * 8 + warp; item < items; item += (int64_t)gridDim.x * 8) {
    const int t = static_cast<int>(item / heads), hd = static_cast<int>(item % heads);
    const bool isq = hd < nh;
    const int h = isq ? hd : hd - nh;
    const int col = isq ? h * d : nh * d + h * d;
    const bf16* xs = qkv + (int64_t)t * ld + col;
    const float* gs = isq ? dq + (int64_t)t * nh * d + h * d : dk + (int64_t)t * nkv * d + h * d;
    const float* g = isq ? gq : gk;
    const float r = isq ? rq[(int64_t)t * nh + h] : rk[(int64_t)t * nkv + h];
    const int pos = t % S;
    float xh[2][2][2], dxh[2][2][2];
    float dot = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int i = 2 * lane + 64 * j;
      if (i < half) {
        const uint32_t a = *reinterpret_cast<const uint32_t*>(xs + i);
        const uint32_t b = *reinterpret_cast<const uint32_t*>(xs + half + i);
        const float2 d0 = *reinterpret_cast<const float2*>(gs + i);
        const float2 d1 = *reinterpret_cast<const float2*>(gs + half + i);
        const float in0[2] = {d0.x, d0.y}, in1[2] = {d1.x, d1.y};
        const float xv0[2] = {bf16lo(a), bf16hi(a)}, xv1[2] = {bf16lo(b), bf16hi(b)};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float2 c = cs[(int64_t)pos * half + i + e];
          const float dn0 = in0[e] * c.x + in1[e] * c.y;  // inverse rotation
          const float dn1 = in1[e] * c.x - in0[e] * c.y;
          xh[j][0][e] = xv0[e] * r;
          xh[j][1][e] = xv1[e] * r;
          // gain gradient contributions
          if (isq) {
            accq[j][0][e] += dn0 * xh[j][0][e];
            accq[j][1][e] += dn1 * xh[j][1][e];
          } else {
            acck[j][0][e] += dn0 * xh[j][0][e];
            acck[j][1][e] += dn1 * xh[j][1][e];
          }
          dxh[j][0][e] = dn0 * g[i + e];
          dxh[j][1][e] = dn1 * g[half + i + e];
          dot += dxh[j][0][e] * xh[j][0][e] + dxh[j][1][e] * xh[j][1][e];
        }
      }
    }
    const float cmean = warp_sum(dot) / d;
    bf16* out = dqkv + (int64_t)t * ld + col;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int i = 2 * lane + 64 * j;
      if (i < half) {
        float o[2][2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int e = 0; e < 2; ++e) o[hh][e] = r * (dxh[j][hh][e] - xh[j][hh][e] * cmean);
        *reinterpret_cast<uint32_t*>(out + i) = pack_bf16x2(o[0][0], o[0][1]);
        *reinterpret_cast<uint32_t*>(out + half + i) = pack_bf16x2(o[1][0], o[1][1]);
      }
    }
  }
  // per-warp partials to shared memory, then a fixed-order sum over warps
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int i = 2 * lane + 64 * j;
    if (i < half) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          red[warp][0][hh * half + i + e] = accq[j][hh][e];
          red[warp][1][hh * half + i + e] = acck[j][hh][e];
        }
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < 2 * d; c += blockDim.x) {
    const int which = c / d, i = c % d;
    float sum = 0.f;
    for (int w = 0; w < 8; ++w) sum += red[w][which][i];
    partials[(int64_t)blockIdx.x * 2 * d + c] = sum;
  }
}

int qknorm_bwd_partial_rows(int T, int heads) {
  const int64_t want = ((int64_t)T * heads + 7) / 8;
  const int cap = min(2 * num_sms(), kMaxPartialRows);
  return want < cap ? static_cast<int>(want) : cap;
}

cudaError_t qknorm_rope_bwd(const float* dq, const float* dk, const bf16* qkv, int64_t ld_qkv,
                            const float* rstd_q, const float* rstd_k, const float* gq,
                            const float* gk, const float* cs, bf16* dqkv, float* dg_qk,
                            float* partials, int T, int S, int nh, int nkv, int d,
                            cudaStream_t s) {
  const int P = qknorm_bwd_partial_rows(T, nh + nkv);
  note_launch();
  qknorm_rope_bwd_kernel<<<P, 256, 0, s>>>(dq, dk, qkv, ld_qkv, rstd_q, rstd_k, gq, gk,
                                           reinterpret_cast<const float2*>(cs), dqkv, partials, T,
                                           S, nh, nkv, d);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // columns [0, d) -> q gain, [d, 2d) -> k gain
  note_launch();
  reduce_cols_kernel<<<1, 256, 0, s>>>(partials, P, 2 * d, dg_qk);
  return cudaGetLastError();
}

// --------------------------------------------------------------------- cast
__global__ void cast_bf16_kernel(const float4* __restrict__ src, uint2* __restrict__ dst,
                                 int64_t n4) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 v = src[i];
    dst[i] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
  }
}
__global__ void cast_bf16_tail_kernel(const float* __restrict__ src, bf16* __restrict__ dst,
                                      int64_t start, int64_t n) {
  const int64_t i = start + threadIdx.x;
  if (i < n) dst[i] = __float2bfloat16_rn(src[i]);
}

cudaError_t cast_bf16(const float* src, bf16* dst, int64_t n, cudaStream_t s) {
  const int64_t n4 = n / 4;
  if (n4 > 0) {
    int64_t blocks = (n4 + 255) / 256;
    const int64_t cap = 8LL * num_sms();
    if (blocks > cap) blocks = cap;
    note_launch();
    cast_bf16_kernel<<<(unsigned)blocks, 256, 0, s>>>(reinterpret_cast<const float4*>(src),
                                                      reinterpret_cast<uint2*>(dst), n4);
  }
  if (n % 4) {
    note_launch();
    cast_bf16_tail_kernel<<<1, 32, 0, s>>>(src, dst, n4 * 4, n);
  }
  return cudaGetLastError();
}

// -------------------------------------------------------------- CE finalise
// lse[t] = log-sum-exp over the per-tile (max, sum exp) partials;
// loss[t] = lse[t] - z[t, target[t]] (the target logit kept in fp32).
__global__ void ce_finalize_kernel(const float2* __restrict__ part, int part_ld, int ntiles,
                                   const float* __restrict__ tgt, float* __restrict__ lse,
                                   float* __restrict__ loss, int T) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= T) return;
  const float2* p = part + (int64_t)row * part_ld;
  float m = -INFINITY;
  for (int i = lane; i < ntiles; i += 32) m = fmaxf(m, p[i].x);
  m = warp_max(m);
  float s = 0.f;
  for (int i = lane; i < ntiles; i += 32) s += p[i].y * __expf(p[i].x - m);
  s = warp_sum(s);
  if (lane == 0) {
    const float l = m + logf(s);
    lse[row] = l;
    loss[row] = l - tgt[row];
  }
}

cudaError_t ce_finalize(const float2* part, int part_ld, int ntiles, const float* tgt_logit,
                        float* lse, float* loss, int T, cudaStream_t s) {
  note_launch();
  ce_finalize_kernel<<<(T + 7) / 8, 256, 0, s>>>(part, part_ld, ntiles, tgt_logit, lse, loss, T);
  return cudaGetLastError();
}

// dz = (exp(z - lse) - onehot(target)) * scale, in place over the bf16 logits.
__global__ void ce_grad_kernel(uint4* __restrict__ z, const float* __restrict__ lse,
                               const int32_t* __restrict__ targets, float scale, int T, int V8) {
  const int64_t n = (int64_t)T * V8;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int row = static_cast<int>(i / V8);
    const int c0 = static_cast<int>(i % V8) * 8;
    const float l = lse[row];
    const int tg = targets[row];
    uint4 v = z[i];
    uint32_t* w = &v.x;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float a = __expf(bf16lo(w[k]) - l);
      float b = __expf(bf16hi(w[k]) - l);
      if (c0 + 2 * k == tg) a -= 1.f;
      if (c0 + 2 * k + 1 == tg) b -= 1.f;
      w[k] = pack_bf16x2(a * scale, b * scale);
    }
    z[i] = v;
  }
}

cudaError_t ce_grad(bf16* z, const float* lse, const int32_t* targets, float scale, int T, int V,
                    cudaStream_t s) {
  const int V8 = V / 8;
  const int64_t n = (int64_t)T * V8;
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = 8LL * num_sms();
  if (blocks > cap) blocks = cap;
  note_launch();
  ce_grad_kernel<<<(unsigned)blocks, 256, 0, s>>>(reinterpret_cast<uint4*>(z), lse, targets, scale,
                                                  T, V8);
  return cudaGetLastError();
}

// -------------------------------------------------------------- squared sum
constexpr int kMaxBufs = 64;
struct BufTable {
  const float* p[kMaxBufs];
  int64_t n[kMaxBufs];
  int nbuf;
};

// Per-thread: fp32 over 8 elements, fp64 across those groups; block: fp64
// tree; partials[block] written, summed in block order by sq_sum_final.
__global__ void __launch_bounds__(256) sq_sum_kernel(const BufTable tab,
                                                     double* __restrict__ partials) {
  __shared__ double red[8];
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  double acc = 0.0;
  for (int b = 0; b < tab.nbuf; ++b) {
    const float* p = tab.p[b];
    const int64_t n = tab.n[b];
    const int64_t n8 = n / 8;
    const float4* p4 = reinterpret_cast<const float4*>(p);
    for (int64_t i = tid; i < n8; i += nthr) {
      const float4 a = p4[2 * i], c = p4[2 * i + 1];
      float s = a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w;
      s += c.x * c.x + c.y * c.y + c.z * c.z + c.w * c.w;
      acc += static_cast<double>(s);
    }
    for (int64_t i = n8 * 8 + tid; i < n; i += nthr) {
      const float v = p[i];
      acc += static_cast<double>(v * v);
    }
  }
  acc = warp_sum_d(acc);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int w = 0; w < 8; ++w) s += red[w];
    partials[blockIdx.x] = s;
  }
}

__global__ void sq_sum_final_kernel(const double* __restrict__ partials, int P,
                                    double* __restrict__ out) {
  __shared__ double red[256];
  double s = 0.0;
  for (int i = threadIdx.x; i < P; i += 256) s += partials[i];
  red[threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int i = 0; i < 256; ++i) t += red[i];
    *out = t;
  }
}

cudaError_t sq_sum(const float* const* bufs, const int64_t* lens, int nbuf, double* out,
                   double* partials, int max_partials, cudaStream_t s) {
  BufTable tab;
  int64_t total = 0;
  tab.nbuf = nbuf;
  for (int i = 0; i < nbuf; ++i) {
    tab.p[i] = bufs[i];
    tab.n[i] = lens[i];
    total += lens[i];
  }
  int64_t blocks = (total / 8 + 255) / 256;
  if (blocks < 1) blocks = 1;
  const int64_t cap = 4LL * num_sms();
  if (blocks > cap) blocks = cap;
  if (blocks > max_partials) blocks = max_partials;
  note_launch();
  sq_sum_kernel<<<(unsigned)blocks, 256, 0, s>>>(tab, partials);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  note_launch();
  sq_sum_final_kernel<<<1, 256, 0, s>>>(partials, (int)blocks, out);
  return cudaGetLastError();
}

// --------------------------------------------------------------- clip scale
__global__ void clip_scale_kernel(const double* __restrict__ sumsq, float max_norm,
                                  float* __restrict__ scale, int32_t* __restrict__ nonfinite) {
  const double norm = sqrt(*sumsq);
  const bool finite = isfinite(norm);
  float sc = 1.0f;
  if (finite && norm > static_cast<double>(max_norm))
    sc = static_cast<float>(static_cast<double>(max_norm) / norm);
  *scale = sc;
  if (nonfinite) *nonfinite = finite ? 0 : 1;
}

cudaError_t clip_scale(const double* sumsq, float max_norm, float* scale, int32_t* nonfinite,
                       cudaStream_t s) {
  note_launch();
  clip_scale_kernel<<<1, 1, 0, s>>>(sumsq, max_norm, scale, nonfinite);
  return cudaGetLastError();
}

// -------------------------------------------------------------------- AdamW
__device__ __forceinline__ float adamw_one(float& w, float g, float& m, float& v, float sc,
                                           float lr, float b1, float b2, float eps, float wd,
                                           float bc1, float bc2) {
  const float gs = sc * g;
  m = b1 * m + (1.0f - b1) * gs;
  v = b2 * v + (1.0f - b2) * gs * gs;
  const float mhat = m / bc1;
  const float vhat = v / bc2;
  w = w - lr * (mhat / (sqrtf(vhat) + eps) + wd * w);
  return w;
}

__global__ void __launch_bounds__(256) adamw_kernel(float4* __restrict__ w,
                                                    const float4* __restrict__ g,
                                                    float4* __restrict__ m, float4* __restrict__ v,
                                                    int64_t n4, const float* __restrict__ scale,
                                                    const int32_t* __restrict__ skip, float lr,
                                                    float b1, float b2, float eps, float wd,
                                                    float bc1, float bc2, uint2* __restrict__ wb) {
  if (skip && *skip) return;
  const float sc = scale ? *scale : 1.0f;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    float4 wv = w[i], mv = m[i], vv = v[i];
    const float4 gv = g[i];
    adamw_one(wv.x, gv.x, mv.x, vv.x, sc, lr, b1, b2, eps, wd, bc1, bc2);
    adamw_one(wv.y, gv.y, mv.y, vv.y, sc, lr, b1, b2, eps, wd, bc1, bc2);
    adamw_one(wv.z, gv.z, mv.z, vv.z, sc, lr, b1, b2, eps, wd, bc1, bc2);
    adamw_one(wv.w, gv.w, mv.w, vv.w, sc, lr, b1, b2, eps, wd, bc1, bc2);
    w[i] = wv;
    m[i] = mv;
    v[i] = vv;
    if (wb) wb[i] = make_uint2(pack_bf16x2(wv.x, wv.y), pack_bf16x2(wv.z, wv.w));
  }
}

__global__ void adamw_tail_kernel(float* __restrict__ w, const float* __restrict__ g,
                                  float* __restrict__ m, float* __restrict__ v, int64_t start,
                                  int64_t n, const float* __restrict__ scale,
                                  const int32_t* __restrict__ skip, float lr, float b1, float b2,
                                  float eps, float wd, float bc1, float bc2, bf16* __restrict__ wb) {
  if (skip && *skip) return;
  const int64_t i = start + threadIdx.x;
  if (i >= n) return;
  const float sc = scale ? *scale : 1.0f;
  float wv = w[i], mv = m[i], vv = v[i];
  adamw_one(wv, g[i], mv, vv, sc, lr, b1, b2, eps, wd, bc1, bc2);
  w[i] = wv;
  m[i] = mv;
  v[i] = vv;
  if (wb) wb[i] = __float2bfloat16_rn(wv);
}

cudaError_t adamw(float* w, const float* g, float* m, float* v, int64_t n, const float* scale,
                  const int32_t* skip, float lr, float b1, float b2, float eps, float wd,
                  float bc1, float bc2, bf16* wb, cudaStream_t s) {
  const int64_t n4 = n / 4;
  if (n4 > 0) {
    int64_t blocks = (n4 + 255) / 256;
    const int64_t cap = 8LL * num_sms();
    if (blocks > cap) blocks = cap;
    note_launch();
    adamw_kernel<<<(unsigned)blocks, 256, 0, s>>>(
        reinterpret_cast<float4*>(w), reinterpret_cast<const float4*>(g),
        reinterpret_cast<float4*>(m), reinterpret_cast<float4*>(v), n4, scale, skip, lr, b1, b2,
        eps, wd, bc1, bc2, reinterpret_cast<uint2*>(wb));
  }
  if (n % 4) {
    note_launch();
    adamw_tail_kernel<<<1, 32, 0, s>>>(w, g, m, v, n4 * 4, n, scale, skip, lr, b1, b2, eps, wd,
                                       bc1, bc2, wb);
  }
  return cudaGetLastError();
}

}  // namespace rdt
