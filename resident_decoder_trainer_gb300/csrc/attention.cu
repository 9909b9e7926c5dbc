// Causal grouped-query flash attention, forward and backward (bf16 operands,
// fp32 softmax and accumulation) on mma.sync tiles, for the small head_dim 16
// and 32; head_dim 64 and 128 run on the tcgen05 kernels (attention_tc.cu).
//
// Forward: one CTA per (128-query tile, query head, sequence); 8 warps own 16
// query rows each; K/V tiles of 64 keys stream through a cp.async double
// buffer; the scores never leave registers (online softmax in the log2
// domain) and the log-sum-exp of every row is saved for the backward.
// Query head h reads kv head h / (nh/nkv) straight from the token-major
// projection buffers, so no head expansion, transpose or layout copy exists.
//
// Backward: one CTA per (64-key tile, kv head, sequence) loops over the
// nh/nkv query heads of its group and over the query tiles at or below the
// diagonal. dK and dV of the whole group accumulate in registers (the GQA
// reduction is free); dQ is accumulated into an fp32 buffer with vector
// reductions, so its last bits depend on the order the CTAs run in.
#include "common.cuh"
#include "internal.h"

namespace rdt {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct AttnSmem {
  static constexpr int LD = D + 8;  // padded row (bf16 elements): conflict-free ldmatrix
};

// Copy `rows` x D bf16 rows (global row stride ld elements) into padded smem,
// zero-filling rows at or beyond `valid`.
template <int D, int ROWS, int NTHREADS>
__device__ __forceinline__ void load_tile(uint32_t dst, const bf16* src, int64_t ld, int valid) {
  constexpr int CHUNKS = D / 8;  // 16-byte chunks per row
  constexpr int LD = D + 8;
#pragma unroll
  for (int i = threadIdx.x; i < ROWS * CHUNKS; i += NTHREADS) {
    const int r = i / CHUNKS, c = i % CHUNKS;
    const bool ok = r < valid;
    const bf16* g = src + (ok ? (int64_t)r * ld : 0) + c * 8;
    cp_async16(dst + (r * LD + c * 8) * 2, g, ok);
  }
}

}  // namespace

// --------------------------------------------------------------- forward
template <int D>
__global__ void __launch_bounds__(256) attn_fwd_kernel(const bf16* __restrict__ q, int64_t ldq,
                                                       const bf16* __restrict__ k, int64_t ldk,
                                                       const bf16* __restrict__ v, int64_t ldv,
                                                       bf16* __restrict__ o, float* __restrict__ lse,
                                                       int S, int nh, int nkv, float scale_log2) {
  constexpr int BM = 128, BNK = 64, LD = D + 8;
  extern __shared__ __align__(16) uint8_t smem[];
  bf16* Qs = reinterpret_cast<bf16*>(smem);
  bf16* Ks = Qs + BM * LD;   // [2][BNK][LD]
  bf16* Vs = Ks + 2 * BNK * LD;  // [2][BNK][LD]

  const int mt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = h / (nh / nkv);
  const int m0 = mt * BM;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t tok0 = (int64_t)b * S;

  const bf16* qb = q + (tok0 + m0) * ldq + h * D;
  const bf16* kb = k + tok0 * ldk + g * D;
  const bf16* vb = v + tok0 * ldv + g * D;

  const int n_tiles = min((S + BNK - 1) / BNK, (m0 + BM + BNK - 1) / BNK);

  load_tile<D, BM, 256>(smem_u32(Qs), qb, ldq, S - m0);
  load_tile<D, BNK, 256>(smem_u32(Ks), kb, ldk, S);
  load_tile<D, BNK, 256>(smem_u32(Vs), vb, ldv, S);
  cp_async_commit();

  uint32_t qf[D / 16][4];
  float oacc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

  const int gq = lane >> 2, tq = lane & 3;
  const int row_a = m0 + warp * 16 + gq;  // query positions of this thread's two rows
  const int row_b = row_a + 8;

  for (int j = 0; j < n_tiles; ++j) {
    if (j + 1 < n_tiles) {
      const int n1 = (j + 1) * BNK;
      load_tile<D, BNK, 256>(smem_u32(Ks + ((j + 1) & 1) * BNK * LD), kb + (int64_t)n1 * ldk, ldk,
                             S - n1);
      load_tile<D, BNK, 256>(smem_u32(Vs + ((j + 1) & 1) * BNK * LD), vb + (int64_t)n1 * ldv, ldv,
                             S - n1);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (j == 0) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int r = warp * 16 + (lane & 15), c = kk * 16 + 8 * (lane >> 4);
        ldsm_x4(smem_u32(Qs + r * LD + c), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
      }
    }
    const int n0 = j * BNK;
    // this warp's rows all precede the tile: nothing to do
    if (n0 <= m0 + warp * 16 + 15) {
      const bf16* Kt = Ks + (j & 1) * BNK * LD;
      const bf16* Vt = Vs + (j & 1) * BNK * LD;
      float s[BNK / 8][4];
#pragma unroll
      for (int i = 0; i < BNK / 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int np = 0; np < BNK / 16; ++np) {
          uint32_t b0, b1, b2, b3;
          const int r = np * 16 + (lane & 7) + 8 * (lane >> 4);
          const int c = kk * 16 + 8 * ((lane >> 3) & 1);
          ldsm_x4(smem_u32(Kt + r * LD + c), b0, b1, b2, b3);
          mma_16816(s[2 * np], qf[kk], b0, b1);
          mma_16816(s[2 * np + 1], qf[kk], b2, b3);
        }
      }
      // mask, scale into the log2 domain, online softmax
      float mx[2] = {mrow[0], mrow[1]};
#pragma unroll
      for (int i = 0; i < BNK / 8; ++i) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int col = n0 + i * 8 + 2 * tq + (e & 1);
          const int row = (e < 2) ? row_a : row_b;
          float x = s[i][e] * scale_log2;
          if (col > row || col >= S) x = -INFINITY;
          s[i][e] = x;
          mx[e >> 1] = fmaxf(mx[e >> 1], x);
        }
      }
#pragma unroll
      for (int r2 = 0; r2 < 2; ++r2) {
        mx[r2] = fmaxf(mx[r2], __shfl_xor_sync(0xffffffffu, mx[r2], 1));
        mx[r2] = fmaxf(mx[r2], __shfl_xor_sync(0xffffffffu, mx[r2], 2));
      }
      float alpha[2];
#pragma unroll
      for (int r2 = 0; r2 < 2; ++r2) {
        alpha[r2] = (mrow[r2] == -INFINITY) ? 0.f : exp2f(mrow[r2] - mx[r2]);
        mrow[r2] = mx[r2];
        lrow[r2] *= alpha[r2];
      }
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        oacc[i][0] *= alpha[0];
        oacc[i][1] *= alpha[0];
        oacc[i][2] *= alpha[1];
        oacc[i][3] *= alpha[1];
      }
#pragma unroll
      for (int i = 0; i < BNK / 8; ++i) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float m = mrow[e >> 1];
          const float p = (s[i][e] == -INFINITY) ? 0.f : exp2f(s[i][e] - m);
          s[i][e] = p;
          lrow[e >> 1] += p;
        }
      }
      // O += P V
#pragma unroll
      for (int kk = 0; kk < BNK / 16; ++kk) {
        uint32_t a[4];
        a[0] = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
        a[1] = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
        a[2] = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        a[3] = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
        for (int dn = 0; dn < D / 16; ++dn) {
          uint32_t b0, b1, b2, b3;
          const int r = kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
          const int c = dn * 16 + 8 * (lane >> 4);
          ldsm_x4_t(smem_u32(Vt + r * LD + c), b0, b1, b2, b3);
          mma_16816(oacc[2 * dn], a, b0, b1);
          mma_16816(oacc[2 * dn + 1], a, b2, b3);
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

#pragma unroll
  for (int r2 = 0; r2 < 2; ++r2) {
    lrow[r2] += __shfl_xor_sync(0xffffffffu, lrow[r2], 1);
    lrow[r2] += __shfl_xor_sync(0xffffffffu, lrow[r2], 2);
  }
  const float inv[2] = {lrow[0] > 0.f ? 1.f / lrow[0] : 0.f, lrow[1] > 0.f ? 1.f / lrow[1] : 0.f};
#pragma unroll
  for (int r2 = 0; r2 < 2; ++r2) {
    const int row = r2 ? row_b : row_a;
    if (row >= S) continue;
    bf16* orow = o + (tok0 + row) * (int64_t)(nh * D) + h * D;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      const uint32_t pk = pack_bf16x2(oacc[i][2 * r2] * inv[r2], oacc[i][2 * r2 + 1] * inv[r2]);
      *reinterpret_cast<uint32_t*>(orow + i * 8 + 2 * tq) = pk;
    }
    if (tq == 0) lse[((int64_t)b * nh + h) * S + row] = (mrow[r2] + log2f(lrow[r2])) * kLn2;
  }
}

// ------------------------------------------------------ backward: D = rowsum(dO o O)
// d/8 lanes per (token, head) item, 16 bytes of each operand per lane; each
// thread takes kPreRounds items spaced one grid apart, so every round streams
// one contiguous stretch of O and dO, with all loads issued before the first
// product. Writes D[(b*nh + h)*S_ld + s] and, if lse2 is given, lse2 (same
// index) = lse[(b*nh + h)*S + s] * log2(e); positions S <= s < S_ld get 0 in
// both, so the padded segments the tensor-core backward reads are finite.
constexpr int kPreRounds = 4;

template <int D>
__global__ void __launch_bounds__(256) attn_bwd_pre_kernel(const bf16* __restrict__ o,
                                                           const bf16* __restrict__ dout,
                                                           const float* __restrict__ lse,
                                                           float* __restrict__ Dd,
                                                           float* __restrict__ lse2, int B, int S,
                                                           int S_ld, int nh) {
  constexpr int L = D / 8;  // lanes per item
  const int items = B * S * nh;
  const int g = static_cast<int>(blockIdx.x) * 256 + static_cast<int>(threadIdx.x);
  const int stride = static_cast<int>(gridDim.x) * (256 / L);  // items per round
  const int base = g / L, sub = g % L;
  uint4 a[kPreRounds], c[kPreRounds];
#pragma unroll
  for (int r = 0; r < kPreRounds; ++r) {
    const int it = base + r * stride;
    if (it < items) {
      const int64_t off = static_cast<int64_t>(it) * D + 8 * sub;
      a[r] = *reinterpret_cast<const uint4*>(o + off);
      c[r] = *reinterpret_cast<const uint4*>(dout + off);
    } else {
      a[r] = make_uint4(0u, 0u, 0u, 0u);
      c[r] = a[r];
    }
  }
#pragma unroll
  for (int r = 0; r < kPreRounds; ++r) {
    const uint32_t* pa = &a[r].x;
    const uint32_t* pc = &c[r].x;
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) acc += bf16lo(pa[e]) * bf16lo(pc[e]) + bf16hi(pa[e]) * bf16hi(pc[e]);
#pragma unroll
    for (int off = L / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    const int it = base + r * stride;
    if (sub == 0 && it < items) {
      const int t = it / nh, h = it - t * nh;
      const int b = t / S, s = t - b * S;
      const int64_t bh = static_cast<int64_t>(b) * nh + h;
      Dd[bh * S_ld + s] = acc;
      if (lse2) lse2[bh * S_ld + s] = lse[bh * S + s] * kLog2e;
    }
  }
  // the padding of every (sequence, head) row
  const int pad = S_ld - S;
  for (int i = g; i < B * nh * pad; i += static_cast<int>(gridDim.x) * 256) {
    const int64_t bh = i / pad;
    const int s = S + i % pad;
    Dd[bh * S_ld + s] = 0.f;
    if (lse2) lse2[bh * S_ld + s] = 0.f;
  }
}

// ------------------------------------------------------------ backward main
template <int D>
__global__ void __launch_bounds__(128) attn_bwd_kernel(
    const bf16* __restrict__ q, int64_t ldq, const bf16* __restrict__ k, int64_t ldk,
    const bf16* __restrict__ v, int64_t ldv, const bf16* __restrict__ dout,
    const float* __restrict__ lse, const float* __restrict__ Dd, float* __restrict__ dq,
    float* __restrict__ dk, bf16* __restrict__ dv, int64_t lddv, int S, int nh, int nkv,
    float scale, float scale_log2) {
  constexpr int BKV = 64, BQ = 64, LD = D + 8, LDS = BQ + 8;
  extern __shared__ __align__(16) uint8_t smem[];
  bf16* Ks = reinterpret_cast<bf16*>(smem);
  bf16* Vs = Ks + BKV * LD;
  bf16* Qs = Vs + BKV * LD;      // [2][BQ][LD]
  bf16* dOs = Qs + 2 * BQ * LD;  // [2][BQ][LD]
  bf16* dSs = dOs + 2 * BQ * LD;  // [BKV][LDS]
  float* Ls = reinterpret_cast<float*>(dSs + BKV * LDS);  // [2][BQ] lse (log2 domain)
  float* Ds = Ls + 2 * BQ;                                // [2][BQ]

  const int nt = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int rep = nh / nkv;
  const int n0 = nt * BKV;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int64_t tok0 = (int64_t)b * S;

  load_tile<D, BKV, 128>(smem_u32(Ks), k + (tok0 + n0) * ldk + g * D, ldk, S - n0);
  load_tile<D, BKV, 128>(smem_u32(Vs), v + (tok0 + n0) * ldv + g * D, ldv, S - n0);

  const int q_tiles = (S + BQ - 1) / BQ;
  const int first_qt = n0 / BQ;
  const int per_head = q_tiles - first_qt;
  const int iters = rep * per_head;

  auto issue = [&](int it, int buf) {
    const int hh = g * rep + it / per_head;
    const int m0 = (first_qt + it % per_head) * BQ;
    load_tile<D, BQ, 128>(smem_u32(Qs + buf * BQ * LD), q + (tok0 + m0) * ldq + hh * D, ldq, S - m0);
    load_tile<D, BQ, 128>(smem_u32(dOs + buf * BQ * LD), dout + (tok0 + m0) * (int64_t)(nh * D) + hh * D,
                          nh * D, S - m0);
    for (int i = threadIdx.x; i < BQ; i += 128) {
      const int row = m0 + i;
      const int64_t idx = ((int64_t)b * nh + hh) * S + row;
      Ls[buf * BQ + i] = row < S ? lse[idx] * kLog2e : INFINITY;
      Ds[buf * BQ + i] = row < S ? Dd[idx] : 0.f;
    }
  };

  float dka[D / 8][4], dva[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) dka[i][e] = dva[i][e] = 0.f;

  if (iters > 0) issue(0, 0);
  cp_async_commit();

  const int kv_a = n0 + warp * 16 + gq;  // this thread's two key positions
  const int kv_b = kv_a + 8;

  for (int it = 0; it < iters; ++it) {
    const int buf = it & 1;
    const int hh = g * rep + it / per_head;
    const int m0 = (first_qt + it % per_head) * BQ;
    if (it + 1 < iters) issue(it + 1, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const bf16* Qt = Qs + buf * BQ * LD;
    const bf16* dOt = dOs + buf * BQ * LD;
    const float* Lt = Ls + buf * BQ;
    const float* Dt = Ds + buf * BQ;

    // S^T = K Q^T and dP^T = V dO^T for this warp's 16 keys x 64 queries
    float st[BQ / 8][4], dpt[BQ / 8][4];
#pragma unroll
    for (int i = 0; i < BQ / 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) st[i][e] = dpt[i][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t ka[4], va[4];
      {
        const int r = warp * 16 + (lane & 15), c = kk * 16 + 8 * (lane >> 4);
        ldsm_x4(smem_u32(Ks + r * LD + c), ka[0], ka[1], ka[2], ka[3]);
        ldsm_x4(smem_u32(Vs + r * LD + c), va[0], va[1], va[2], va[3]);
      }
#pragma unroll
      for (int np = 0; np < BQ / 16; ++np) {
        const int r = np * 16 + (lane & 7) + 8 * (lane >> 4);
        const int c = kk * 16 + 8 * ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_u32(Qt + r * LD + c), b0, b1, b2, b3);
        mma_16816(st[2 * np], ka, b0, b1);
        mma_16816(st[2 * np + 1], ka, b2, b3);
        ldsm_x4(smem_u32(dOt + r * LD + c), b0, b1, b2, b3);
        mma_16816(dpt[2 * np], va, b0, b1);
        mma_16816(dpt[2 * np + 1], va, b2, b3);
      }
    }
    // P^T and dS^T = P^T o (dP^T - D)
#pragma unroll
    for (int i = 0; i < BQ / 8; ++i) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int qi = i * 8 + 2 * tq + (e & 1);
        const int qrow = m0 + qi;
        const int key = (e < 2) ? kv_a : kv_b;
        float p = exp2f(st[i][e] * scale_log2 - Lt[qi]);
        if (qrow < key || qrow >= S || key >= S) p = 0.f;
        st[i][e] = p;
        dpt[i][e] = p * (dpt[i][e] - Dt[qi]);
      }
    }
    // dV += P^T dO, dK += dS^T Q
#pragma unroll
    for (int kk = 0; kk < BQ / 16; ++kk) {
      uint32_t pa[4], da[4];
      pa[0] = pack_bf16x2(st[2 * kk][0], st[2 * kk][1]);
      pa[1] = pack_bf16x2(st[2 * kk][2], st[2 * kk][3]);
      pa[2] = pack_bf16x2(st[2 * kk + 1][0], st[2 * kk + 1][1]);
      pa[3] = pack_bf16x2(st[2 * kk + 1][2], st[2 * kk + 1][3]);
      da[0] = pack_bf16x2(dpt[2 * kk][0], dpt[2 * kk][1]);
      da[1] = pack_bf16x2(dpt[2 * kk][2], dpt[2 * kk][3]);
      da[2] = pack_bf16x2(dpt[2 * kk + 1][0], dpt[2 * kk + 1][1]);
      da[3] = pack_bf16x2(dpt[2 * kk + 1][2], dpt[2 * kk + 1][3]);
#pragma unroll
      for (int dn = 0; dn < D / 16; ++dn) {
        const int r = kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int c = dn * 16 + 8 * (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_u32(dOt + r * LD + c), b0, b1, b2, b3);
        mma_16816(dva[2 * dn], pa, b0, b1);
        mma_16816(dva[2 * dn + 1], pa, b2, b3);
        ldsm_x4_t(smem_u32(Qt + r * LD + c), b0, b1, b2, b3);
        mma_16816(dka[2 * dn], da, b0, b1);
        mma_16816(dka[2 * dn + 1], da, b2, b3);
      }
      // stage dS^T (bf16) for the dQ product
      const int c0 = kk * 16 + 2 * tq;
      const int ra = warp * 16 + gq;
      *reinterpret_cast<uint32_t*>(dSs + ra * LDS + c0) = da[0];
      *reinterpret_cast<uint32_t*>(dSs + (ra + 8) * LDS + c0) = da[1];
      *reinterpret_cast<uint32_t*>(dSs + ra * LDS + c0 + 8) = da[2];
      *reinterpret_cast<uint32_t*>(dSs + (ra + 8) * LDS + c0 + 8) = da[3];
    }
    __syncthreads();
    // dQ[64 q, D] += scale * dS K: warp w owns query rows 16w..16w+15
    {
      uint32_t af[BKV / 16][4];
#pragma unroll
      for (int kk = 0; kk < BKV / 16; ++kk) {
        const int r = kk * 16 + (lane & 7) + 8 * (lane >> 4);
        const int c = warp * 16 + 8 * ((lane >> 3) & 1);
        ldsm_x4_t(smem_u32(dSs + r * LDS + c), af[kk][0], af[kk][1], af[kk][2], af[kk][3]);
      }
      const int qa = m0 + warp * 16 + gq, qb = qa + 8;
      float* dqa = dq + (tok0 + qa) * (int64_t)(nh * D) + hh * D;
      float* dqb = dqa + 8 * (int64_t)(nh * D);
#pragma unroll
      for (int dn = 0; dn < D / 16; ++dn) {
        float acc[2][4];
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[0][e] = acc[1][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk) {
          const int r = kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
          const int c = dn * 16 + 8 * (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(smem_u32(Ks + r * LD + c), b0, b1, b2, b3);
          mma_16816(acc[0], af[kk], b0, b1);
          mma_16816(acc[1], af[kk], b2, b3);
        }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int col = dn * 16 + hf * 8 + 2 * tq;
          if (qa < S)
            asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(dqa + col),
                         "f"(acc[hf][0] * scale), "f"(acc[hf][1] * scale)
                         : "memory");
          if (qb < S)
            asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(dqb + col),
                         "f"(acc[hf][2] * scale), "f"(acc[hf][3] * scale)
                         : "memory");
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  // write dK (fp32, scaled) and dV (bf16)
#pragma unroll
  for (int r2 = 0; r2 < 2; ++r2) {
    const int key = r2 ? kv_b : kv_a;
    if (key >= S) continue;
    float* dkr = dk + (tok0 + key) * (int64_t)(nkv * D) + g * D;
    bf16* dvr = dv + (tok0 + key) * lddv + g * D;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      const int col = i * 8 + 2 * tq;
      *reinterpret_cast<float2*>(dkr + col) =
          make_float2(dka[i][2 * r2] * scale, dka[i][2 * r2 + 1] * scale);
      *reinterpret_cast<uint32_t*>(dvr + col) = pack_bf16x2(dva[i][2 * r2], dva[i][2 * r2 + 1]);
    }
  }
}

// -------------------------------------------------------------------- host
template <int D>
static size_t fwd_smem() {
  return (size_t)(128 + 4 * 64) * (D + 8) * 2;
}
template <int D>
static size_t bwd_smem() {
  return (size_t)(2 * 64 + 4 * 64) * (D + 8) * 2 + 64 * (64 + 8) * 2 + 4 * 64 * 4;
}

template <int D>
static cudaError_t fwd_d(const bf16* q, int64_t ldq, const bf16* k, int64_t ldk, const bf16* v,
                         int64_t ldv, bf16* o, float* lse, int B, int S, int nh, int nkv,
                         cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)fwd_smem<D>());
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid((S + 127) / 128, nh, B);
  const float scale_log2 = kLog2e / sqrtf((float)D);
  note_launch();
  attn_fwd_kernel<D><<<grid, 256, fwd_smem<D>(), s>>>(q, ldq, k, ldk, v, ldv, o, lse, S, nh, nkv,
                                                       scale_log2);
  return cudaGetLastError();
}

template <int D>
static cudaError_t bwd_d(const bf16* q, int64_t ldq, const bf16* k, int64_t ldk, const bf16* v,
                         int64_t ldv, const bf16* dout, const float* lse, const float* Dd,
                         float* dq, float* dk, bf16* dv, int64_t lddv, int B, int S, int nh,
                         int nkv, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)bwd_smem<D>());
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid((S + 63) / 64, nkv, B);
  const float scale = 1.0f / sqrtf((float)D);
  note_launch();
  attn_bwd_kernel<D><<<grid, 128, bwd_smem<D>(), s>>>(q, ldq, k, ldk, v, ldv, dout, lse, Dd, dq, dk,
                                                       dv, lddv, S, nh, nkv, scale,
                                                       scale * kLog2e);
  return cudaGetLastError();
}

cudaError_t attn_fwd(const bf16* q, int64_t ldq, const bf16* k, int64_t ldk, const bf16* v,
                     int64_t ldv, bf16* o, float* lse, int B, int S, int nh, int nkv, int d,
                     cudaStream_t s) {
  switch (d) {
    case 16: return fwd_d<16>(q, ldq, k, ldk, v, ldv, o, lse, B, S, nh, nkv, s);
    case 32: return fwd_d<32>(q, ldq, k, ldk, v, ldv, o, lse, B, S, nh, nkv, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t attn_bwd_pre(const bf16* o, const bf16* dout, const float* lse, float* Dd,
                         float* lse2, int B, int S, int S_ld, int nh, int d, cudaStream_t s) {
  const int64_t threads = (int64_t)B * S * nh * (d / 8);
  if (threads >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;  // 32-bit thread indices
  const int per_block = 256 * kPreRounds;
  const dim3 grid(static_cast<unsigned>((threads + per_block - 1) / per_block));
  note_launch();
  switch (d) {
    case 16: attn_bwd_pre_kernel<16><<<grid, 256, 0, s>>>(o, dout, lse, Dd, lse2, B, S, S_ld, nh); break;
    case 32: attn_bwd_pre_kernel<32><<<grid, 256, 0, s>>>(o, dout, lse, Dd, lse2, B, S, S_ld, nh); break;
    case 64: attn_bwd_pre_kernel<64><<<grid, 256, 0, s>>>(o, dout, lse, Dd, lse2, B, S, S_ld, nh); break;
    case 128: attn_bwd_pre_kernel<128><<<grid, 256, 0, s>>>(o, dout, lse, Dd, lse2, B, S, S_ld, nh); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t attn_bwd(const bf16* q, int64_t ldq, const bf16* k, int64_t ldk, const bf16* v,
                     int64_t ldv, const bf16* dout, const float* lse, const float* Dd, float* dq,
                     float* dk, bf16* dv, int64_t lddv, int B, int S, int nh, int nkv, int d,
                     cudaStream_t s) {
  switch (d) {
    case 16: return bwd_d<16>(q, ldq, k, ldk, v, ldv, dout, lse, Dd, dq, dk, dv, lddv, B, S, nh, nkv, s);
    case 32: return bwd_d<32>(q, ldq, k, ldk, v, ldv, dout, lse, Dd, dq, dk, dv, lddv, B, S, nh, nkv, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace rdt
