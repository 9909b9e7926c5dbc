// Causal grouped-query flash attention on the 5th-generation tensor cores
// (tcgen05.mma, TMEM accumulators, TMA-fed shared memory), bf16 operands,
// fp32 softmax and accumulation.
//
// Forward (head_dim 64 or 128): one CTA per (128-query tile, query head,
// sequence), heaviest tiles first. Warp 0 streams Q once and 128-key K/V tiles
// through a 2-stage ring; warp 1 issues S = Q K^T into one of two TMEM score
// buffers (so the next tile's scores are computed while this tile's softmax
// runs) and O += P V into a TMEM output accumulator; warps 2-5 (one query row
// per thread) run the online softmax in the log2 domain, rescale O in TMEM
// when the row maximum moves, and write P as bf16 into a 128-byte-swizzled
// shared tile that the next MMA reads as its A operand. The log-sum-exp of
// every row is kept for the backward.
//
// Backward (head_dim 128): one CTA per (128-key tile, kv head, sequence) loops
// over the query heads of its group and over 64-query tiles at or below the
// diagonal. Per tile: S^T = K Q^T and dP^T = V dO^T into TMEM; warps 2-5 (one
// key row per thread) form P^T and dS^T = P^T o (dP^T - D) and write both to
// swizzled shared tiles; then dV += P^T dO and dK += dS^T Q accumulate in
// TMEM for the whole group (the GQA reduction costs nothing) and
// dQ^T = K^T dS^T goes to one of two TMEM buffers that warps 6-9 (one head
// dimension per thread) add into the fp32 dQ with coalesced reductions.
// Every operand transposition is a shared-memory descriptor, never a copy.
#include "common.cuh"
#include "internal.h"

namespace rdt {

namespace {
constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kLn2F = 0.6931471805599453f;
}  // namespace

// ============================================================== forward
template <int D>
struct FwdCfg {
  static constexpr int BM = 128, BN = 128;
  static constexpr uint32_t CHUNK = 128 * 128;            // 64 cols x 128 rows of bf16
  static constexpr uint32_t Q_BYTES = BM * D * 2;
  static constexpr uint32_t KV_BYTES = BN * D * 2;
  static constexpr uint32_t P_BYTES = BM * BN * 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;        // [2]
  static constexpr uint32_t OFF_V = OFF_K + 2 * KV_BYTES;   // [2]
  static constexpr uint32_t OFF_P = OFF_V + 2 * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_P + P_BYTES;
  static constexpr size_t SMEM = OFF_BAR + 256 + 1024;
  static constexpr uint32_t TMEM_S = 0, TMEM_O = 256, TMEM_COLS = 512;
};

template <int D>
__global__ void __launch_bounds__(192, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv, bf16* __restrict__ o,
                       float* __restrict__ lse, int S, int nh, int nkv, float scale_log2,
                       int* err) {
  using C = FwdCfg<D>;
  constexpr int BM = C::BM, BN = C::BN, DCH = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  // barriers (8 bytes each)
  const uint32_t q_full = bar0, k_full = bar0 + 8, v_full = bar0 + 24, kv_empty = bar0 + 40,
                 s_full = bar0 + 56, s_free = bar0 + 72, p_full = bar0 + 88, o_done = bar0 + 96,
                 drain = bar0 + 104;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 128);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = gridDim.x - 1 - blockIdx.x;  // heaviest (longest causal row) tiles first
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = h / (nh / nkv);
  const int m0 = mt * BM;
  const int n_tiles = min((S + BN - 1) / BN, mt + 1);
  const int tok0 = b * S;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(k_full + 8 * i, 1);
      mbar_init(v_full + 8 * i, 1);
      mbar_init(kv_empty + 8 * i, 1);
      mbar_init(s_full + 8 * i, 1);
      mbar_init(s_free + 8 * i, 128);
    }
    mbar_init(p_full, 128);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // --------------------------------------------------------- producer
      mbar_arrive_expect_tx(q_full, C::Q_BYTES);
      for (int c = 0; c < DCH; ++c)
        tma_load_2d(sbase + C::OFF_Q + c * C::CHUNK, &tq, q_full, h * D + c * 64, tok0 + m0);
      uint32_t pending = 0;
      bool ok = true;
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!mbar_wait(kv_empty + 8 * st, ph ^ 1, err)) {
          ok = false;
          break;
        }
        const int n0 = j * BN;
        mbar_arrive_expect_tx(k_full + 8 * st, C::KV_BYTES);
        for (int c = 0; c < DCH; ++c)
          tma_load_2d(sbase + C::OFF_K + st * C::KV_BYTES + c * C::CHUNK, &tk, k_full + 8 * st,
                      g * D + c * 64, tok0 + n0);
        mbar_arrive_expect_tx(v_full + 8 * st, C::KV_BYTES);
        for (int c = 0; c < DCH; ++c)
          tma_load_2d(sbase + C::OFF_V + st * C::KV_BYTES + c * C::CHUNK, &tv, v_full + 8 * st,
                      g * D + c * 64, tok0 + n0);
        pending = (pending & ~(3u << (2 * st))) | ((1u | (ph << 1)) << (2 * st));
      }
      if (!ok) {
        for (int st = 0; st < 2; ++st)
          if ((pending >> (2 * st)) & 1u) {
            const uint32_t ph = (pending >> (2 * st + 1)) & 1u;
            mbar_wait(k_full + 8 * st, ph, nullptr);
            mbar_wait(v_full + 8 * st, ph, nullptr);
          }
        mbar_wait(q_full, 0, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------------------- MMA
      constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(BM, D, 0, 1);
      bool ok = mbar_wait(q_full, 0, err);
      auto issue_s = [&](int j) -> bool {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!mbar_wait(k_full + 8 * st, ph, err)) return false;
        if (!mbar_wait(s_free + 8 * (j & 1), ph ^ 1, err)) return false;
        tc_fence_after();
        const uint32_t kb = sbase + C::OFF_K + st * C::KV_BYTES;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t ad = sdesc_sw128(sbase + C::OFF_Q + (k >> 2) * C::CHUNK + (k & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(kb + (k >> 2) * C::CHUNK + (k & 3) * 32, 16, 1024);
          tc_mma_bf16(tmem + C::TMEM_S + (j & 1) * BN, ad, bd, idesc_s, k > 0);
        }
        tc_commit(s_full + 8 * (j & 1));
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; j < n_tiles && ok; ++j) {
        if (j + 1 < n_tiles && !issue_s(j + 1)) {
          ok = false;
          break;
        }
        const int st = j & 1;
        if (!mbar_wait(p_full, j & 1, err) || !mbar_wait(v_full + 8 * st, (j >> 1) & 1, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t vb = sbase + C::OFF_V + st * C::KV_BYTES;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint64_t ad = sdesc_sw128(sbase + C::OFF_P + (k >> 2) * C::CHUNK + (k & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(vb + k * 2048, C::CHUNK, 1024);
          tc_mma_bf16(tmem + C::TMEM_O, ad, bd, idesc_o, (j | k) != 0);
        }
        tc_commit(o_done);
        tc_commit(kv_empty + 8 * st);
      }
      tc_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else {
    // ---------------------------------------------------------- softmax
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int qpos = m0 + row;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    uint8_t* p_tile = smem + C::OFF_P;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      if (!warp_wait(s_full + 8 * (j & 1), (j >> 1) & 1, err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c)
        tmem_ld32(tmem + lane_base + C::TMEM_S + (j & 1) * BN + c * 32,
                  *reinterpret_cast<uint32_t(*)[32]>(&sv[c * 32]));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(s_free + 8 * (j & 1));
      const int n0 = j * BN;
      float mx = m_run;
      const bool diag = (n0 + BN > qpos) || (n0 + BN > S);
#pragma unroll
      for (int c = 0; c < BN; ++c) {
        float x = __uint_as_float(sv[c]) * scale_log2;
        if (diag && (n0 + c > qpos || n0 + c >= S)) x = -INFINITY;
        sv[c] = __float_as_uint(x);
        mx = fmaxf(mx, x);
      }
      const float alpha = (m_run == -INFINITY) ? 0.f : ex2_approx(m_run - mx);
      m_run = mx;
      float sum = 0.f;
      // bf16 pairs of P are packed in place into sv[0 .. BN/2)
#pragma unroll
      for (int c = 0; c < BN; c += 2) {
        const float p0 = ex2_approx(__uint_as_float(sv[c]) - mx);
        const float p1 = ex2_approx(__uint_as_float(sv[c + 1]) - mx);
        sum += p0 + p1;
        sv[c / 2] = pack_bf16x2(p0, p1);
      }
      l_run = l_run * alpha + sum;
      if (j > 0) {
        // O and the P tile are still in use by the previous P V product
        if (!warp_wait(o_done, (j - 1) & 1, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tmem + lane_base + C::TMEM_O + c * 32, ov);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st32(tmem + lane_base + C::TMEM_O + c * 32, ov);
          }
          tmem_st_wait();
        }
      }
      // P row -> swizzled K-major tile (two 64-column chunks)
#pragma unroll
      for (int cc = 0; cc < BN / 8; ++cc) {
        const uint32_t off = (cc >> 3) * C::CHUNK + sw128_offset(row, cc & 7);
        *reinterpret_cast<uint4*>(p_tile + off) =
            make_uint4(sv[4 * cc], sv[4 * cc + 1], sv[4 * cc + 2], sv[4 * cc + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (ok && warp_wait(o_done, (n_tiles - 1) & 1, err)) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      bf16* orow = o + (int64_t)(tok0 + qpos) * (nh * D) + h * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(tmem + lane_base + C::TMEM_O + c * 32, ov);
        tmem_ld_wait();
        if (qpos < S) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(ov[8 * q4 + 0]) * inv, __uint_as_float(ov[8 * q4 + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(ov[8 * q4 + 2]) * inv, __uint_as_float(ov[8 * q4 + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(ov[8 * q4 + 4]) * inv, __uint_as_float(ov[8 * q4 + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(ov[8 * q4 + 6]) * inv, __uint_as_float(ov[8 * q4 + 7]) * inv);
            reinterpret_cast<uint4*>(orow + c * 32)[q4] = v;
          }
        }
      }
      if (qpos < S) lse[((int64_t)b * nh + h) * S + qpos] = (m_run + __log2f(l_run)) * kLn2F;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ============================================================= backward
struct BwdCfg {
  static constexpr int D = 128, BKV = 128, BQ = 64;
  static constexpr uint32_t KV_CHUNK = 128 * 128;  // 64 d-cols x 128 key rows
  static constexpr uint32_t Q_CHUNK = 64 * 128;    // 64 d-cols x 64 query rows
  static constexpr uint32_t KV_BYTES = BKV * D * 2;
  static constexpr uint32_t Q_BYTES = BQ * D * 2;
  static constexpr uint32_t T_BYTES = BKV * BQ * 2;  // P^T / dS^T tiles: 128 rows x 128 B
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + KV_BYTES;
  static constexpr uint32_t OFF_Q = OFF_V + KV_BYTES;      // [2]
  static constexpr uint32_t OFF_DO = OFF_Q + 2 * Q_BYTES;  // [2]
  static constexpr uint32_t OFF_PT = OFF_DO + 2 * Q_BYTES;
  static constexpr uint32_t OFF_DST = OFF_PT + T_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_DST + T_BYTES;
  static constexpr size_t SMEM = OFF_BAR + 256 + 1024;
  // TMEM columns
  static constexpr uint32_t T_DK = 0, T_DV = 128, T_ST = 256, T_DPT = 320, T_DQ = 384;
  static constexpr uint32_t TMEM_COLS = 512;
};

__global__ void __launch_bounds__(320, 1)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                       const float* __restrict__ lse, const float* __restrict__ Dd,
                       float* __restrict__ dq, float* __restrict__ dk, bf16* __restrict__ dv,
                       int64_t lddv, int S, int nh, int nkv, float scale, float scale_log2,
                       int* err) {
  using C = BwdCfg;
  constexpr int D = C::D, BKV = C::BKV, BQ = C::BQ;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t kv_full = bar0, q_full = bar0 + 8, q_empty = bar0 + 24, s_full = bar0 + 40,
                 s_used = bar0 + 48, p_ready = bar0 + 56, pd_free = bar0 + 64,
                 dq_full = bar0 + 72, dq_empty = bar0 + 88, fin = bar0 + 104, drain = bar0 + 112;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 128);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int rep = nh / nkv;
  const int n0 = nt * BKV;
  const int tok0 = b * S;
  const int q_tiles = (S + BQ - 1) / BQ;
  const int first_qt = n0 / BQ;
  const int per_head = q_tiles - first_qt;
  const int iters = rep * per_head;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(q_full + 8 * i, 1);
      mbar_init(q_empty + 8 * i, 1);
      mbar_init(dq_full + 8 * i, 1);
      mbar_init(dq_empty + 8 * i, 128);
    }
    mbar_init(s_full, 1);
    mbar_init(s_used, 128);
    mbar_init(p_ready, 128);
    mbar_init(pd_free, 1);
    mbar_init(fin, 1);
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    tma_prefetch_desc(&tdo);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // --------------------------------------------------------- producer
      mbar_arrive_expect_tx(kv_full, 2 * C::KV_BYTES);
      for (int c = 0; c < 2; ++c) {
        tma_load_2d(sbase + C::OFF_K + c * C::KV_CHUNK, &tk, kv_full, g * D + c * 64, tok0 + n0);
        tma_load_2d(sbase + C::OFF_V + c * C::KV_CHUNK, &tv, kv_full, g * D + c * 64, tok0 + n0);
      }
      uint32_t pending = 0;
      bool ok = true;
      for (int it = 0; it < iters && ok; ++it) {
        const int st = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        if (!mbar_wait(q_empty + 8 * st, ph ^ 1, err)) {
          ok = false;
          break;
        }
        const int hh = g * rep + it / per_head;
        const int m0 = (first_qt + it % per_head) * BQ;
        mbar_arrive_expect_tx(q_full + 8 * st, 2 * C::Q_BYTES);
        for (int c = 0; c < 2; ++c) {
          tma_load_2d(sbase + C::OFF_Q + st * C::Q_BYTES + c * C::Q_CHUNK, &tq, q_full + 8 * st,
                      hh * D + c * 64, tok0 + m0);
          tma_load_2d(sbase + C::OFF_DO + st * C::Q_BYTES + c * C::Q_CHUNK, &tdo,
                      q_full + 8 * st, hh * D + c * 64, tok0 + m0);
        }
        pending = (pending & ~(3u << (2 * st))) | ((1u | (ph << 1)) << (2 * st));
      }
      if (!ok) {
        mbar_wait(kv_full, 0, nullptr);
        for (int st = 0; st < 2; ++st)
          if ((pending >> (2 * st)) & 1u) mbar_wait(q_full + 8 * st, (pending >> (2 * st + 1)) & 1u, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------------------- MMA
      constexpr uint32_t id_s = idesc_bf16_f32(128, BQ, 0, 0);   // S^T, dP^T
      constexpr uint32_t id_kv = idesc_bf16_f32(128, D, 0, 1);   // dV, dK
      constexpr uint32_t id_q = idesc_bf16_f32(128, BQ, 1, 1);   // dQ^T (M = head dim)
      bool ok = mbar_wait(kv_full, 0, err);
      auto issue_s = [&](int it) -> bool {
        const int st = it & 1;
        if (!mbar_wait(q_full + 8 * st, (it >> 1) & 1, err)) return false;
        if (!mbar_wait(s_used, (it & 1) ^ 1, err)) return false;  // S^T/dP^T TMEM consumed
        tc_fence_after();
        const uint32_t qb = sbase + C::OFF_Q + st * C::Q_BYTES;
        const uint32_t ob = sbase + C::OFF_DO + st * C::Q_BYTES;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t koff = (k >> 2) * C::KV_CHUNK + (k & 3) * 32;
          const uint32_t qoff = (k >> 2) * C::Q_CHUNK + (k & 3) * 32;
          tc_mma_bf16(tmem + C::T_ST, sdesc_sw128(sbase + C::OFF_K + koff, 16, 1024),
                      sdesc_sw128(qb + qoff, 16, 1024), id_s, k > 0);
          tc_mma_bf16(tmem + C::T_DPT, sdesc_sw128(sbase + C::OFF_V + koff, 16, 1024),
                      sdesc_sw128(ob + qoff, 16, 1024), id_s, k > 0);
        }
        tc_commit(s_full);
        return true;
      };
      if (ok && iters > 0) ok = issue_s(0);
      for (int it = 0; it < iters && ok; ++it) {
        const int st = it & 1;
        if (it + 1 < iters && !issue_s(it + 1)) {
          ok = false;
          break;
        }
        if (!mbar_wait(p_ready, it & 1, err) ||
            !mbar_wait(dq_empty + 8 * st, ((it >> 1) & 1) ^ 1, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t qb = sbase + C::OFF_Q + st * C::Q_BYTES;
        const uint32_t ob = sbase + C::OFF_DO + st * C::Q_BYTES;
#pragma unroll
        for (int k = 0; k < BQ / 16; ++k) {
          // dV += P^T dO ; dK += dS^T Q   (K = query rows)
          tc_mma_bf16(tmem + C::T_DV, sdesc_sw128(sbase + C::OFF_PT + k * 32, 16, 1024),
                      sdesc_sw128(ob + k * 2048, C::Q_CHUNK, 1024), id_kv, (it | k) != 0);
          tc_mma_bf16(tmem + C::T_DK, sdesc_sw128(sbase + C::OFF_DST + k * 32, 16, 1024),
                      sdesc_sw128(qb + k * 2048, C::Q_CHUNK, 1024), id_kv, (it | k) != 0);
        }
#pragma unroll
        for (int k = 0; k < BKV / 16; ++k) {
          // dQ^T = K^T dS^T   (K = key rows)
          tc_mma_bf16(tmem + C::T_DQ + st * BQ,
                      sdesc_sw128(sbase + C::OFF_K + k * 2048, C::KV_CHUNK, 1024),
                      sdesc_sw128(sbase + C::OFF_DST + k * 2048, C::T_BYTES, 1024), id_q, k > 0);
        }
        tc_commit(pd_free);
        tc_commit(q_empty + 8 * st);
        tc_commit(dq_full + 8 * st);
      }
      tc_commit(fin);
      tc_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else if (warp < 6) {
    // ----------------------------------------------- P^T and dS^T (key rows)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // key row within the tile
    const int kpos = n0 + row;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = true;
    for (int it = 0; it < iters; ++it) {
      const int hh = g * rep + it / per_head;
      const int m0 = (first_qt + it % per_head) * BQ;
      if (!warp_wait(s_full, it & 1, err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[BQ], dp[BQ];
      tmem_ld32(tmem + lane_base + C::T_ST, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      tmem_ld32(tmem + lane_base + C::T_ST + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      tmem_ld32(tmem + lane_base + C::T_DPT, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
      tmem_ld32(tmem + lane_base + C::T_DPT + 32, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(s_used);
      const float* lrow = lse + ((int64_t)b * nh + hh) * S + m0;
      const float* drow = Dd + ((int64_t)b * nh + hh) * S + m0;
      // bf16 pairs of P^T / dS^T are packed in place into sv / dp [0 .. BQ/2)
#pragma unroll
      for (int c = 0; c < BQ; c += 2) {
        float pv[2], dsv[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int qpos = m0 + c + e;
          const bool valid = qpos < S && qpos >= kpos && kpos < S;
          const float l2 = valid ? __ldg(lrow + c + e) * kLog2eF : 0.f;
          const float dd = valid ? __ldg(drow + c + e) : 0.f;
          const float p = valid ? ex2_approx(__uint_as_float(sv[c + e]) * scale_log2 - l2) : 0.f;
          pv[e] = p;
          dsv[e] = p * (__uint_as_float(dp[c + e]) - dd);
        }
        sv[c / 2] = pack_bf16x2(pv[0], pv[1]);
        dp[c / 2] = pack_bf16x2(dsv[0], dsv[1]);
      }
      if (it > 0 && !warp_wait(pd_free, (it - 1) & 1, err)) {
        ok = false;
        break;
      }
      uint8_t* pt = smem + C::OFF_PT;
      uint8_t* dst = smem + C::OFF_DST;
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        const uint32_t off = sw128_offset(row, c8);
        *reinterpret_cast<uint4*>(pt + off) =
            make_uint4(sv[4 * c8], sv[4 * c8 + 1], sv[4 * c8 + 2], sv[4 * c8 + 3]);
        *reinterpret_cast<uint4*>(dst + off) =
            make_uint4(dp[4 * c8], dp[4 * c8 + 1], dp[4 * c8 + 2], dp[4 * c8 + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_ready);
    }
    // dK (scaled) and dV of this key tile, summed over the query heads of the group
    if (ok && warp_wait(fin, 0, err)) {
      tc_fence_after();
      float* dkr = dk + (int64_t)(tok0 + kpos) * (nkv * D) + g * D;
      bf16* dvr = dv + (int64_t)(tok0 + kpos) * lddv + g * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t a[32], v[32];
        tmem_ld32(tmem + lane_base + C::T_DK + c * 32, a);
        tmem_ld32(tmem + lane_base + C::T_DV + c * 32, v);
        tmem_ld_wait();
        if (kpos < S) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            reinterpret_cast<float4*>(dkr + c * 32)[e] =
                make_float4(__uint_as_float(a[4 * e]) * scale, __uint_as_float(a[4 * e + 1]) * scale,
                            __uint_as_float(a[4 * e + 2]) * scale, __uint_as_float(a[4 * e + 3]) * scale);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            reinterpret_cast<uint4*>(dvr + c * 32)[e] = make_uint4(
                pack_bf16x2(__uint_as_float(v[8 * e]), __uint_as_float(v[8 * e + 1])),
                pack_bf16x2(__uint_as_float(v[8 * e + 2]), __uint_as_float(v[8 * e + 3])),
                pack_bf16x2(__uint_as_float(v[8 * e + 4]), __uint_as_float(v[8 * e + 5])),
                pack_bf16x2(__uint_as_float(v[8 * e + 6]), __uint_as_float(v[8 * e + 7])));
        }
      }
    }
  } else {
    // ------------------------------------------- dQ (one head dim per thread)
    const int quarter = warp & 3;
    const int dcol = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    for (int it = 0; it < iters; ++it) {
      const int st = it & 1;
      const int hh = g * rep + it / per_head;
      const int m0 = (first_qt + it % per_head) * BQ;
      if (!warp_wait(dq_full + 8 * st, (it >> 1) & 1, err)) break;
      tc_fence_after();
      uint32_t qv[BQ];
      tmem_ld32(tmem + lane_base + C::T_DQ + st * BQ, *reinterpret_cast<uint32_t(*)[32]>(&qv[0]));
      tmem_ld32(tmem + lane_base + C::T_DQ + st * BQ + 32, *reinterpret_cast<uint32_t(*)[32]>(&qv[32]));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(dq_empty + 8 * st);
      float* base = dq + (int64_t)(tok0 + m0) * (nh * D) + hh * D + dcol;
      const int nq = min(BQ, S - m0);
#pragma unroll
      for (int c = 0; c < BQ; ++c)
        if (c < nq)
          asm volatile("red.global.add.f32 [%0], %1;" ::"l"(base + (int64_t)c * (nh * D)),
                       "f"(__uint_as_float(qv[c]) * scale)
                       : "memory");
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ================================================================== host
template <int D>
static cudaError_t fwd_tc_d(const bf16* q, int64_t ldq, const bf16* k, int64_t ldk, const bf16* v,
                            int64_t ldv, bf16* o, float* lse, int B, int S, int nh, int nkv,
                            int* err, cudaStream_t s) {
  const int64_t T = (int64_t)B * S;
  CUtensorMap tq, tk, tv;
  if (!make_tma_2d(&tq, q, T, (int64_t)nh * D, ldq, 128) ||
      !make_tma_2d(&tk, k, T, (int64_t)nkv * D, ldk, 128) ||
      !make_tma_2d(&tv, v, T, (int64_t)nkv * D, ldv, 128))
    return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)FwdCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid((S + 127) / 128, nh, B);
  const float scale_log2 = kLog2eF / sqrtf((float)D);
  note_launch();
  attn_fwd_tc_kernel<D><<<grid, 192, FwdCfg<D>::SMEM, s>>>(tq, tk, tv, o, lse, S, nh, nkv,
                                                           scale_log2, err);
  return cudaGetLastError();
}

bool attn_tc_supported(int d, bool backward) { return backward ? d == 128 : (d == 64 || d == 128); }

cudaError_t attn_fwd_tc(const bf16* q, int64_t ldq, const bf16* k, int64_t ldk, const bf16* v,
                        int64_t ldv, bf16* o, float* lse, int B, int S, int nh, int nkv, int d,
                        int* err, cudaStream_t s) {
  if (d == 128) return fwd_tc_d<128>(q, ldq, k, ldk, v, ldv, o, lse, B, S, nh, nkv, err, s);
  if (d == 64) return fwd_tc_d<64>(q, ldq, k, ldk, v, ldv, o, lse, B, S, nh, nkv, err, s);
  return cudaErrorInvalidValue;
}

cudaError_t attn_bwd_tc(const bf16* q, int64_t ldq, const bf16* k, int64_t ldk, const bf16* v,
                        int64_t ldv, const bf16* dout, const float* lse, const float* Dd,
                        float* dq, float* dk, bf16* dv, int64_t lddv, int B, int S, int nh,
                        int nkv, int d, int* err, cudaStream_t s) {
  if (d != 128) return cudaErrorInvalidValue;
  constexpr int D = 128;
  const int64_t T = (int64_t)B * S;
  CUtensorMap tq, tk, tv, tdo;
  if (!make_tma_2d(&tq, q, T, (int64_t)nh * D, ldq, 64) ||
      !make_tma_2d(&tk, k, T, (int64_t)nkv * D, ldk, 128) ||
      !make_tma_2d(&tv, v, T, (int64_t)nkv * D, ldv, 128) ||
      !make_tma_2d(&tdo, dout, T, (int64_t)nh * D, (int64_t)nh * D, 64))
    return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)BwdCfg::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid((S + 127) / 128, nkv, B);
  const float scale = 1.0f / sqrtf((float)D);
  note_launch();
  attn_bwd_tc_kernel<<<grid, 320, BwdCfg::SMEM, s>>>(tq, tk, tv, tdo, lse, Dd, dq, dk, dv, lddv, S,
                                                     nh, nkv, scale, scale * kLog2eF, err);
  return cudaGetLastError();
}

}  // namespace rdt
