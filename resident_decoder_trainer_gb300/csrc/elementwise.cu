// HBM-bound kernels of the training step: RMSNorm forward/backward (with the
// residual add and deterministic gain-gradient reduction), per-head QK
// RMSNorm + RoPE-neox forward/backward, the merge of the LM head's
// per-chunk cross-entropy statistics, the multi-buffer squared sum, the clip
// scale and AdamW. All are single-pass (or two-pass where a row statistic is
// needed), 128-bit vectorised, with warp-shuffle reductions; every reduction
// runs in a fixed order, so results are bitwise reproducible run to run.
#include <cmath>

#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

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

// dx = r*(dy*g - xhat*mean(dy*g*xhat)) + resid, single pass over the row.
// One CTA per group of rows; thread t owns columns [8t, 8t+8) for every row
// (so its gain-gradient partial needs no cross-thread reduction); the row
// dot product is a warp shuffle + a fixed-order sum over the CTA's warps.
__global__ void __launch_bounds__(512) rmsnorm_bwd_kernel(
    const float* __restrict__ dy, const float* __restrict__ x, const float* __restrict__ rstd,
    const float* __restrict__ gamma, const float* __restrict__ resid, float* __restrict__ dx,
    bf16* __restrict__ dxb, float* __restrict__ partials, int T, int H) {
  __shared__ float red[2][16];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int c0 = 8 * threadIdx.x;
  const bool own = c0 < H;
  float g[8], acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = g[e] = 0.f;  // idle lanes must add exact zeros
  if (own) {
    const float4 g0 = *reinterpret_cast<const float4*>(gamma + c0);
    const float4 g1 = *reinterpret_cast<const float4*>(gamma + c0 + 4);
    g[0] = g0.x; g[1] = g0.y; g[2] = g0.z; g[3] = g0.w;
    g[4] = g1.x; g[5] = g1.y; g[6] = g1.z; g[7] = g1.w;
  }
  const float invH = 1.0f / H;
  int buf = 0;
  for (int row = blockIdx.x; row < T; row += gridDim.x) {
    const int64_t base = (int64_t)row * H + c0;
    float a[8] = {}, b[8] = {}, q[8] = {};
    if (own) {
      const float4 a0 = *reinterpret_cast<const float4*>(dy + base);
      const float4 a1 = *reinterpret_cast<const float4*>(dy + base + 4);
      const float4 b0 = *reinterpret_cast<const float4*>(x + base);
      const float4 b1 = *reinterpret_cast<const float4*>(x + base + 4);
      a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
      a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
      b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
      b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
      if (resid) {
        const float4 q0 = *reinterpret_cast<const float4*>(resid + base);
        const float4 q1 = *reinterpret_cast<const float4*>(resid + base + 4);
        q[0] = q0.x; q[1] = q0.y; q[2] = q0.z; q[3] = q0.w;
        q[4] = q1.x; q[5] = q1.y; q[6] = q1.z; q[7] = q1.w;
      }
    }
    const float r = rstd[row];
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) dot += a[e] * g[e] * b[e];
    dot = warp_sum(dot);
    if (lane == 0) red[buf][warp] = dot;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < nwarps; ++w) tot += red[buf][w];
    buf ^= 1;
    const float cmean = tot * r * invH;  // mean(dy*g*xhat)
    if (own) {
      float o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float xh = b[e] * r;
        o[e] = r * (a[e] * g[e] - xh * cmean) + q[e];
        acc[e] += a[e] * xh;
      }
      *reinterpret_cast<float4*>(dx + base) = make_float4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<float4*>(dx + base + 4) = make_float4(o[4], o[5], o[6], o[7]);
      if (dxb)
        *reinterpret_cast<uint4*>(dxb + base) =
            make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]),
                       pack_bf16x2(o[4], o[5]), pack_bf16x2(o[6], o[7]));
    }
  }
  if (own) {
    float* pr = partials + (int64_t)blockIdx.x * H + c0;
    *reinterpret_cast<float4*>(pr) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4*>(pr + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// out[c] (= or, with accumulate, +=) sum_p partials[p, c]. A cluster of
// `split` CTAs (1..8) serves 32 columns: CTA r of the cluster sums the rows
// p = r*8 + ty, r*8 + ty + 8*split, ... (8 row-strided sums per column, added
// in order), and CTA 0 adds the split CTAs' column sums in rank order, read
// through distributed shared memory. Deterministic for a given split.
constexpr int kRcMaxSplit = 8;
__global__ void __launch_bounds__(256) reduce_cols_kernel(const float* __restrict__ partials,
                                                          int P, int W, float* __restrict__ out,
                                                          int accumulate) {
  __shared__ float red[8][33];
  __shared__ float part[kRcMaxSplit][32];
  cg::cluster_group cl = cg::this_cluster();
  const int split = static_cast<int>(cl.num_blocks());
  const int r = static_cast<int>(cl.block_rank());
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + tx;
  float s = 0.f;
  if (c < W)
    for (int p = r * 8 + ty; p < P; p += 8 * split) s += partials[(int64_t)p * W + c];
  red[ty][tx] = s;
  __syncthreads();
  if (ty == 0) {
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) t += red[i][tx];
    cl.map_shared_rank(&part[0][0], 0)[r * 32 + tx] = t;
  }
  cl.sync();  // the column sums have landed in CTA 0; no CTA leaves before
  if (r == 0 && ty == 0 && c < W) {
    float t = 0.f;
    for (int q = 0; q < split; ++q) t += part[q][tx];
    out[c] = accumulate ? out[c] + t : t;
  }
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

// CTAs (= partial rows) of rmsnorm_bwd: one per row up to one full wave, the
// resident CTAs of all SMs (the row loop is uniform, so a second partial wave
// would only add a tail), within kMaxPartialRows.
int rmsnorm_bwd_partial_rows(int T, int threads) {
  static int per_sm[17] = {};  // by threads / 32 (threads <= 512)
  const int w = threads / 32;
  if (w < 1 || w > 16) return 1;
  if (per_sm[w] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, rmsnorm_bwd_kernel, threads, 0) !=
            cudaSuccess || n < 1)
      n = 1;
    per_sm[w] = n;
  }
  int cap = per_sm[w] * num_sms();
  if (cap > kMaxPartialRows) cap = kMaxPartialRows / num_sms() * num_sms();
  if (cap < 1) cap = 1;
  return T < cap ? (T > 0 ? T : 1) : cap;
}

static cudaError_t reduce_cols(const float* partials, int P, int W, float* out, cudaStream_t s,
                               bool accumulate) {
  // about two CTAs per SM, the rows split over up to 8 CTAs per column block
  const int ncol = (W + 31) / 32;
  int split = (2 * num_sms() + ncol - 1) / ncol;
  if (split > kRcMaxSplit) split = kRcMaxSplit;
  if (split > (P + 7) / 8) split = (P + 7) / 8;
  if (split < 1) split = 1;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(ncol), static_cast<unsigned>(split), 1);
  lc.blockDim = dim3(256, 1, 1);
  lc.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 1;
  at[0].val.clusterDim.y = static_cast<unsigned>(split);
  at[0].val.clusterDim.z = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  note_launch();
  return cudaLaunchKernelEx(&lc, reduce_cols_kernel, partials, P, W, out, accumulate ? 1 : 0);
}

cudaError_t rmsnorm_bwd(const float* dy, const float* x, const float* rstd, const float* gamma,
                        const float* resid, float* dx, bf16* dx_bf16, float* dgamma,
                        float* partials, int T, int H, cudaStream_t s, bool accumulate) {
  const int threads = ((H / 8 + 31) / 32) * 32;
  const int P = rmsnorm_bwd_partial_rows(T, threads);
  note_launch();
  rmsnorm_bwd_kernel<<<P, threads, 0, s>>>(dy, x, rstd, gamma, resid, dx, dx_bf16, partials, T, H);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return reduce_cols(partials, P, H, dgamma, s, accumulate);
}

// ----------------------------------------------------------------- RoPE table
// cs[s, i] = (cos, sin)(s * inv_freq[i]) with inv_freq[i] = theta^(-2i/d)
// computed in fp64 on the host; the angle is formed and reduced modulo 2*pi
// in fp64, then evaluated with the fp32 sincosf on |r| <= pi (+ rounding).
struct InvFreq {
  double v[64];
};
__global__ void rope_table_kernel(float2* __restrict__ cs, int S, int half, const InvFreq f) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= S * half) return;
  const int s = idx / half, i = idx % half;
  const double two_pi = 6.283185307179586476925286766559;
  const double inv_two_pi = 0.15915494309189533576888376337251;
  const double ang = static_cast<double>(s) * f.v[i];
  // nearest multiple of 2 pi; off by one only where ang / (2 pi) sits within
  // rounding of a half-integer, and then |r| is still about pi
  const double k = rint(ang * inv_two_pi);
  const float rr = static_cast<float>(fma(-k, two_pi, ang));
  float sn, cn;
  sincosf(rr, &sn, &cn);
  cs[idx] = make_float2(cn, sn);
}

cudaError_t rope_table(float* cs, int S, int d, float theta, cudaStream_t s) {
  const int half = d / 2;
  InvFreq f;
  for (int i = 0; i < half && i < 64; ++i)
    f.v[i] = std::pow(static_cast<double>(theta), -2.0 * i / d);
  const int n = S * half;
  note_launch();
  rope_table_kernel<<<(n + 255) / 256, 256, 0, s>>>(reinterpret_cast<float2*>(cs), S, half, f);
  return cudaGetLastError();
}

// ----------------------------------------------------- QK RMSNorm + RoPE fwd
// A head of D elements is handled by D/4 lanes, 4 consecutive elements each
// (16-byte fp32 loads); a warp covers 128/D heads per pass. Lanes of the first
// half of a head hold elements i < D/2, their partner (lane ^ D/8) the
// rotation partners i + D/2. A CTA walks whole tokens: every lane loads the
// cos/sin of its 4 rotation pairs once per token and reuses them for all of
// the token's heads; each warp keeps two head groups of loads in flight.
// Heads: nh query heads, nkv key heads, nkv value heads (value heads are only
// converted to bf16 for the attention).
template <int D>
__global__ void __launch_bounds__(256) qknorm_rope_fwd_kernel(
    const float* __restrict__ qkv, int64_t ld, bf16* __restrict__ qo, bf16* __restrict__ ko,
    bf16* __restrict__ vo, float* __restrict__ rq, float* __restrict__ rk,
    const float* __restrict__ gq, const float* __restrict__ gk, const float2* __restrict__ cs,
    int T, int S, int nh, int nkv, float eps) {
  constexpr int LPH = D / 4, HPW = 32 / LPH, PX = LPH / 2, HALF = D / 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot = lane / LPH, sub = lane % LPH;
  const bool first = sub < PX;
  const int i0 = 4 * (first ? sub : sub - PX);
  const int heads = nh + 2 * nkv;
  const int groups = (heads + HPW - 1) / HPW;
  const float4 gq4 = reinterpret_cast<const float4*>(gq)[sub];
  const float4 gk4 = reinterpret_cast<const float4*>(gk)[sub];
  auto head_out = [&](int t, int hd, const float4& xin, const float4& c01, const float4& c23) {
    const bool valid = hd < heads;
    const bool isq = hd < nh;
    const bool isv = hd >= nh + nkv;
    const float x[4] = {xin.x, xin.y, xin.z, xin.w};
    if (valid && isv)
      *reinterpret_cast<uint2*>(vo + ((int64_t)t * nkv + (hd - nh - nkv)) * D + 4 * sub) =
          make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
    float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
#pragma unroll
    for (int o = LPH / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = rsqrtf(ss / D + eps);
    const float4 g4 = isq ? gq4 : gk4;
    const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
    float y[4], yp[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) y[e] = x[e] * r * gv[e];
#pragma unroll
    for (int e = 0; e < 4; ++e) yp[e] = __shfl_xor_sync(0xffffffffu, y[e], PX);
    const float cv[4] = {c01.x, c01.z, c23.x, c23.z}, sv[4] = {c01.y, c01.w, c23.y, c23.w};
    float out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      out[e] = first ? y[e] * cv[e] - yp[e] * sv[e] : y[e] * cv[e] + yp[e] * sv[e];
    if (valid && !isv) {
      bf16* dst = isq ? qo + ((int64_t)t * nh + hd) * D : ko + ((int64_t)t * nkv + (hd - nh)) * D;
      *reinterpret_cast<uint2*>(dst + 4 * sub) =
          make_uint2(pack_bf16x2(out[0], out[1]), pack_bf16x2(out[2], out[3]));
      if (sub == 0) {
        if (isq) rq[(int64_t)t * nh + hd] = r;
        else rk[(int64_t)t * nkv + (hd - nh)] = r;
      }
    }
  };
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    const float4* c4 = reinterpret_cast<const float4*>(cs + (int64_t)(t % S) * HALF + i0);
    const float4 c01 = c4[0], c23 = c4[1];
    const float* row = qkv + (int64_t)t * ld + 4 * sub;
    // three heads' loads in flight per warp
    for (int g0 = warp; g0 < groups; g0 += 24) {
      float4 x[3];
#pragma unroll
      for (int u = 0; u < 3; ++u) {
        const int hu = (g0 + 8 * u) * HPW + slot;
        x[u] = hu < heads ? *reinterpret_cast<const float4*>(row + hu * D)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 3; ++u)
        if (g0 + 8 * u < groups) head_out(t, (g0 + 8 * u) * HPW + slot, x[u], c01, c23);
    }
  }
}

cudaError_t qknorm_rope_fwd(const float* qkv, int64_t ld_qkv, bf16* q_out, bf16* k_out,
                            bf16* v_out, float* rstd_q, float* rstd_k, const float* gq,
                            const float* gk, const float* cs, int T, int S, int nh, int nkv, int d,
                            float eps, cudaStream_t s) {
  const int grid = T < 8 * num_sms() ? (T > 0 ? T : 1) : 8 * num_sms();
  const float2* c2 = reinterpret_cast<const float2*>(cs);
  note_launch();
  switch (d) {
    case 16: qknorm_rope_fwd_kernel<16><<<grid, 256, 0, s>>>(qkv, ld_qkv, q_out, k_out, v_out, rstd_q, rstd_k, gq, gk, c2, T, S, nh, nkv, eps); break;
    case 32: qknorm_rope_fwd_kernel<32><<<grid, 256, 0, s>>>(qkv, ld_qkv, q_out, k_out, v_out, rstd_q, rstd_k, gq, gk, c2, T, S, nh, nkv, eps); break;
    case 64: qknorm_rope_fwd_kernel<64><<<grid, 256, 0, s>>>(qkv, ld_qkv, q_out, k_out, v_out, rstd_q, rstd_k, gq, gk, c2, T, S, nh, nkv, eps); break;
    case 128: qknorm_rope_fwd_kernel<128><<<grid, 256, 0, s>>>(qkv, ld_qkv, q_out, k_out, v_out, rstd_q, rstd_k, gq, gk, c2, T, S, nh, nkv, eps); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// ----------------------------------------------------- QK RMSNorm + RoPE bwd
// Same lane layout and token walk as the forward. Inverse rotation of the
// incoming fp32 gradient, then the RMSNorm backward over head_dim. Gain
// gradients: each lane always owns the same 4 columns, so it accumulates them
// in registers; lanes of different head slots are combined by shuffles, warps
// in a fixed order, and each CTA writes one partial row [q gains | k gains].
template <int D>
__global__ void __launch_bounds__(256, 3) qknorm_rope_bwd_kernel(
    const float* __restrict__ dq, const float* __restrict__ dk, const float* __restrict__ qkv,
    int64_t ld, const float* __restrict__ rq, const float* __restrict__ rk,
    const float* __restrict__ gq, const float* __restrict__ gk, const float2* __restrict__ cs,
    bf16* __restrict__ dqkv, float* __restrict__ partials, int T, int S, int nh, int nkv) {
  constexpr int LPH = D / 4, HPW = 32 / LPH, PX = LPH / 2, HALF = D / 2;
  __shared__ float red[8][2 * D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot = lane / LPH, sub = lane % LPH;
  const bool first = sub < PX;
  const int i0 = 4 * (first ? sub : sub - PX);
  const int heads = nh + nkv;
  const int groups = (heads + HPW - 1) / HPW;
  float accq[4] = {}, acck[4] = {};
  struct In {
    float4 d, x;
    float r;
  };
  auto load = [&](int t, int hd) {
    In in{make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f), 0.f};
    if (hd < heads) {
      const bool isq = hd < nh;
      const float* gsrc = isq ? dq + ((int64_t)t * nh + hd) * D : dk + ((int64_t)t * nkv + (hd - nh)) * D;
      in.d = *reinterpret_cast<const float4*>(gsrc + 4 * sub);
      in.x = *reinterpret_cast<const float4*>(qkv + (int64_t)t * ld + hd * D + 4 * sub);
      in.r = isq ? rq[(int64_t)t * nh + hd] : rk[(int64_t)t * nkv + (hd - nh)];
    }
    return in;
  };
  auto head_grad = [&](int t, int hd, const In& in, const float4& c01, const float4& c23) {
    const bool valid = hd < heads;
    const bool isq = hd < nh;
    const float din[4] = {in.d.x, in.d.y, in.d.z, in.d.w};
    const float xv[4] = {in.x.x, in.x.y, in.x.z, in.x.w};
    float dp[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) dp[e] = __shfl_xor_sync(0xffffffffu, din[e], PX);
    const float cv[4] = {c01.x, c01.z, c23.x, c23.z}, sv[4] = {c01.y, c01.w, c23.y, c23.w};
    const float4 g4 = reinterpret_cast<const float4*>(isq ? gq : gk)[sub];  // L1-resident
    const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
    float xh[4], dxh[4];
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      // inverse rotation: first half d0 c + d1 s, second half d1 c - d0 s
      const float dn = first ? din[e] * cv[e] + dp[e] * sv[e] : din[e] * cv[e] - dp[e] * sv[e];
      xh[e] = xv[e] * in.r;
      if (valid) {
        if (isq) accq[e] += dn * xh[e];
        else acck[e] += dn * xh[e];
      }
      dxh[e] = dn * gv[e];
      dot += dxh[e] * xh[e];
    }
#pragma unroll
    for (int o = LPH / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    const float cmean = dot / D;
    if (valid) {
      float o4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) o4[e] = in.r * (dxh[e] - xh[e] * cmean);
      *reinterpret_cast<uint2*>(dqkv + (int64_t)t * ld + hd * D + 4 * sub) =
          make_uint2(pack_bf16x2(o4[0], o4[1]), pack_bf16x2(o4[2], o4[3]));
    }
  };
  // a warp takes head groups warp, warp + 8, ...: all of a token's loads
  // (up to MAXJ groups) are issued before any is used, so each warp keeps
  // several rows of both inputs in flight
  constexpr int MAXJ = 5;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    const float4* c4 = reinterpret_cast<const float4*>(cs + (int64_t)(t % S) * HALF + i0);
    const float4 c01 = c4[0], c23 = c4[1];
    for (int gb = warp; gb < groups; gb += 8 * MAXJ) {
      In in[MAXJ];
#pragma unroll
      for (int j = 0; j < MAXJ; ++j) {
        const int gi = gb + 8 * j;
        in[j] = load(t, gi < groups ? gi * HPW + slot : heads);
      }
#pragma unroll
      for (int j = 0; j < MAXJ; ++j) {
        const int gi = gb + 8 * j;
        if (gi < groups) head_grad(t, gi * HPW + slot, in[j], c01, c23);  // warp-uniform
      }
    }
  }
  // combine head slots of the warp (lanes with equal sub), fixed order
#pragma unroll
  for (int o = LPH; o < 32; o <<= 1) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      accq[e] += __shfl_xor_sync(0xffffffffu, accq[e], o);
      acck[e] += __shfl_xor_sync(0xffffffffu, acck[e], o);
    }
  }
  if (slot == 0) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      red[warp][4 * sub + e] = accq[e];
      red[warp][D + 4 * sub + e] = acck[e];
    }
  }
  __syncthreads();
  for (int cidx = threadIdx.x; cidx < 2 * D; cidx += blockDim.x) {
    float sum = 0.f;
    for (int w = 0; w < 8; ++w) sum += red[w][cidx];
    partials[(int64_t)blockIdx.x * 2 * D + cidx] = sum;
  }
}

int qknorm_bwd_partial_rows(int T, int) {
  // one CTA (and one partial row) per token up to a whole number of CTAs per
  // SM (3, the kernel's occupancy by its launch bounds) within
  // kMaxPartialRows, so every SM gets the same share of tokens
  int per_sm = kMaxPartialRows / num_sms();
  if (per_sm > 3) per_sm = 3;
  const int cap = per_sm >= 1 ? per_sm * num_sms() : kMaxPartialRows;
  return T < cap ? (T > 0 ? T : 1) : cap;
}

cudaError_t qknorm_rope_bwd(const float* dq, const float* dk, const float* qkv, int64_t ld_qkv,
                            const float* rstd_q, const float* rstd_k, const float* gq,
                            const float* gk, const float* cs, bf16* dqkv, float* dg_qk,
                            float* partials, int T, int S, int nh, int nkv, int d,
                            cudaStream_t s, bool accumulate) {
  const int P = qknorm_bwd_partial_rows(T, nh + nkv);
  const float2* c2 = reinterpret_cast<const float2*>(cs);
  note_launch();
  switch (d) {
    case 16: qknorm_rope_bwd_kernel<16><<<P, 256, 0, s>>>(dq, dk, qkv, ld_qkv, rstd_q, rstd_k, gq, gk, c2, dqkv, partials, T, S, nh, nkv); break;
    case 32: qknorm_rope_bwd_kernel<32><<<P, 256, 0, s>>>(dq, dk, qkv, ld_qkv, rstd_q, rstd_k, gq, gk, c2, dqkv, partials, T, S, nh, nkv); break;
    case 64: qknorm_rope_bwd_kernel<64><<<P, 256, 0, s>>>(dq, dk, qkv, ld_qkv, rstd_q, rstd_k, gq, gk, c2, dqkv, partials, T, S, nh, nkv); break;
    case 128: qknorm_rope_bwd_kernel<128><<<P, 256, 0, s>>>(dq, dk, qkv, ld_qkv, rstd_q, rstd_k, gq, gk, c2, dqkv, partials, T, S, nh, nkv); break;
    default: return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // columns [0, d) -> q gain, [d, 2d) -> k gain
  return reduce_cols(partials, P, 2 * d, dg_qk, s, accumulate);
}

// ----------------------------------------------------- fused squared sums
// One CTA: fixed per-thread strides and a fixed tree, so the result is the
// same bits on every run.
struct SmallBufs {
  const float* p[4];
  int64_t n[4];
};
// Squared-sum slots -> one fp64 total in two launches (latency, not bytes,
// bounds this: ~26 k slots per block backward): kSqCtas CTAs each add a fixed
// slice of the slots and a fixed stride of the gain buffers' squares, then one
// warp adds the kSqCtas partials in index order (deterministic).
__global__ void __launch_bounds__(256) sq_part_kernel(const double* __restrict__ parts,
                                                      int64_t n, const SmallBufs sb, int nsmall,
                                                      double* __restrict__ part2) {
  __shared__ double red[8];
  const int64_t per = (n + kSqCtas - 1) / kSqCtas;
  const int64_t lo = (int64_t)blockIdx.x * per;
  const int64_t hi = lo + per < n ? lo + per : n;
  double acc = 0.0;
  for (int64_t i = lo + threadIdx.x; i < hi; i += 256) acc += parts[i];
  const int64_t gt = (int64_t)blockIdx.x * 256 + threadIdx.x;
  for (int k = 0; k < nsmall; ++k)
    for (int64_t i = gt; i < sb.n[k]; i += (int64_t)kSqCtas * 256) {
      const double v = sb.p[k][i];
      acc += v * v;
    }
  acc = warp_sum_d(acc);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += red[w];
    part2[blockIdx.x] = t;
  }
}

__global__ void __launch_bounds__(32) sq_final2_kernel(const double* __restrict__ part2,
                                                       double* out, int accumulate) {
  double v = part2[threadIdx.x] + part2[threadIdx.x + 32];
  v = warp_sum_d(v);
  if (threadIdx.x == 0) *out = (accumulate ? *out : 0.0) + v;
}

cudaError_t sq_reduce(const double* parts, int64_t n, const float* const* small,
                      const int64_t* small_len, int nsmall, double* out, bool accumulate,
                      double* scratch, cudaStream_t s) {
  if (nsmall < 0 || nsmall > 4 || !scratch) return cudaErrorInvalidValue;
  SmallBufs sb = {};
  for (int i = 0; i < nsmall; ++i) {
    sb.p[i] = small[i];
    sb.n[i] = small_len[i];
  }
  note_launch(2);
  sq_part_kernel<<<kSqCtas, 256, 0, s>>>(parts, n, sb, nsmall, scratch);
  sq_final2_kernel<<<1, 32, 0, s>>>(scratch, out, accumulate ? 1 : 0);
  return cudaGetLastError();
}

// ------------------------------------------------------ LoRA B stacks
struct BPieces {
  const float* p[3];
  int64_t rows[3];
};
__global__ void lora_bstack_kernel(const BPieces bp, int np, int r, int64_t total_rows,
                                   bf16* __restrict__ out) {
  const int64_t cols = static_cast<int64_t>(np) * r;
  const int64_t n = total_rows * cols;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / cols;
    const int col = static_cast<int>(i % cols);
    int64_t off = 0;
    float v = 0.f;
    for (int q = 0; q < np; ++q) {
      if (row >= off && row < off + bp.rows[q]) {
        if (col / r == q) v = bp.p[q][(row - off) * r + col % r];
        break;
      }
      off += bp.rows[q];
    }
    out[i] = __float2bfloat16_rn(v);
  }
}

cudaError_t lora_bstack(const float* const* pieces, const int64_t* rows, int np, int r,
                        bf16* out, cudaStream_t s) {
  if (np < 1 || np > 3 || r < 1) return cudaErrorInvalidValue;
  BPieces bp = {};
  int64_t total = 0;
  for (int q = 0; q < np; ++q) {
    bp.p[q] = pieces[q];
    bp.rows[q] = rows[q];
    total += rows[q];
  }
  const int64_t n = total * np * r;
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = 8LL * num_sms();
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  note_launch();
  lora_bstack_kernel<<<(unsigned)blocks, 256, 0, s>>>(bp, np, r, total, out);
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

// ---------------------------------------------------------------- CE merge
// The log-sum-exp of a row's logits, built chunk by chunk over the vocabulary:
// a chunk's per-tile (max, sum exp) partials are combined around their max,
// then folded into the running (max, sum) of the chunks before it; after the
// last chunk lse = max + log(sum) and loss = lse - z[target] (the target's
// logit kept in fp32 by the chunk that holds it).
__global__ void ce_merge_kernel(const float2* __restrict__ part, int part_ld, int ntiles,
                                float2* __restrict__ run, int first, int last,
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
    if (!first) {
      const float2 r = run[row];
      const float nm = fmaxf(r.x, m);
      s = r.y * __expf(r.x - nm) + s * __expf(m - nm);
      m = nm;
    }
    if (last) {
      const float l = m + logf(s);
      lse[row] = l;
      loss[row] = l - tgt[row];
    } else {
      run[row] = make_float2(m, s);
    }
  }
}

cudaError_t ce_merge(const float2* part, int part_ld, int ntiles, float2* run, bool first,
                     bool last, const float* tgt_logit, float* lse, float* loss, int T,
                     cudaStream_t s) {
  note_launch();
  ce_merge_kernel<<<(T + 7) / 8, 256, 0, s>>>(part, part_ld, ntiles, run, first ? 1 : 0,
                                             last ? 1 : 0, tgt_logit, lse, loss, T);
  return cudaGetLastError();
}

// --------------------------------------------------------------- wait probe
// The bounded-wait error path of the tensor-core kernels, in one warp: it
// holds 32 TMEM columns, waits on an mbarrier (phase 0, one expected arrival)
// with the given limit, and whatever the wait's outcome frees the columns and
// returns. With `arrive` unset nothing ever arrives, so the wait gives up,
// records kErrTimeout in err and the kernel still exits cleanly.
__global__ void __launch_bounds__(32) wait_probe_kernel(int* err, uint64_t limit_ns, int arrive,
                                                        unsigned long long* waited_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_base;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncwarp();
  tmem_alloc(smem_u32(&tmem_base), 32);
  tc_fence_before();
  __syncwarp();
  tc_fence_after();
  const uint32_t taddr = tmem_base;
  if (arrive && threadIdx.x == 0) mbar_arrive(b);
  __syncwarp();
  const uint64_t t0 = global_timer_ns();
  warp_wait(b, 0, err, limit_ns);
  if (threadIdx.x == 0 && waited_ns) *waited_ns = global_timer_ns() - t0;
  tc_fence_before();
  __syncwarp();
  tc_fence_after();
  tmem_dealloc(taddr, 32);
}

cudaError_t wait_probe(int* err, uint64_t limit_ns, bool arrive, unsigned long long* waited_ns,
                       cudaStream_t s) {
  note_launch();
  wait_probe_kernel<<<1, 32, 0, s>>>(err, limit_ns, arrive ? 1 : 0, waited_ns);
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
// 1 - b^step in double, rounded to float (as the host does for a host step).
__device__ __forceinline__ void bias_corrections(int step, float b1, float b2, float& bc1,
                                                 float& bc2) {
  bc1 = static_cast<float>(1.0 - pow(static_cast<double>(b1), static_cast<double>(step)));
  bc2 = static_cast<float>(1.0 - pow(static_cast<double>(b2), static_cast<double>(step)));
}

__global__ void step_advance_kernel(int32_t* step) { *step += 1; }

cudaError_t step_advance(int32_t* step, cudaStream_t s) {
  note_launch();
  step_advance_kernel<<<1, 1, 0, s>>>(step);
  return cudaGetLastError();
}

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
                                                    float bc1, float bc2, uint2* __restrict__ wb,
                                                    const int32_t* __restrict__ step_dev) {
  if (skip && *skip) return;
  const float sc = scale ? *scale : 1.0f;
  if (step_dev) bias_corrections(*step_dev, b1, b2, bc1, bc2);
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
                                  float eps, float wd, float bc1, float bc2, bf16* __restrict__ wb,
                                  const int32_t* __restrict__ step_dev) {
  if (skip && *skip) return;
  const int64_t i = start + threadIdx.x;
  if (i >= n) return;
  const float sc = scale ? *scale : 1.0f;
  if (step_dev) bias_corrections(*step_dev, b1, b2, bc1, bc2);
  float wv = w[i], mv = m[i], vv = v[i];
  adamw_one(wv, g[i], mv, vv, sc, lr, b1, b2, eps, wd, bc1, bc2);
  w[i] = wv;
  m[i] = mv;
  v[i] = vv;
  if (wb) wb[i] = __float2bfloat16_rn(wv);
}

cudaError_t adamw(float* w, const float* g, float* m, float* v, int64_t n, const float* scale,
                  const int32_t* skip, float lr, float b1, float b2, float eps, float wd,
                  float bc1, float bc2, bf16* wb, cudaStream_t s, const int32_t* step_dev) {
  const int64_t n4 = n / 4;
  if (n4 > 0) {
    int64_t blocks = (n4 + 255) / 256;
    const int64_t cap = 8LL * num_sms();
    if (blocks > cap) blocks = cap;
    note_launch();
    adamw_kernel<<<(unsigned)blocks, 256, 0, s>>>(
        reinterpret_cast<float4*>(w), reinterpret_cast<const float4*>(g),
        reinterpret_cast<float4*>(m), reinterpret_cast<float4*>(v), n4, scale, skip, lr, b1, b2,
        eps, wd, bc1, bc2, reinterpret_cast<uint2*>(wb), step_dev);
  }
  if (n % 4) {
    note_launch();
    adamw_tail_kernel<<<1, 32, 0, s>>>(w, g, m, v, n4 * 4, n, scale, skip, lr, b1, b2, eps, wd,
                                       bc1, bc2, wb, step_dev);
  }
  return cudaGetLastError();
}

}  // namespace rdt
