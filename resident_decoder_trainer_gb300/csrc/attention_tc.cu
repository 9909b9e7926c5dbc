// Causal grouped-query flash attention on the 5th-generation tensor cores
// (tcgen05.mma, TMEM accumulators, TMA-fed shared memory), bf16 operands,
// fp32 softmax and accumulation.
//
// Every kernel has 10 warps: warp 0 issues the TMA copies, warp 1 (one lane)
// the tcgen05.mma instructions, and warps 2-9 do the elementwise work: TMEM
// lane quarter q is served by warps 2+q and 6+q (in the backward each takes
// half of the columns of the rows it owns; in the forward each serves its own
// query tile). Work items are launched longest-first (the causal triangle
// makes items unequal).
//
// Forward (head_dim 64 or 128), persistent: each CTA walks work items
// longest first, an item being two 128-query tiles of one head and sequence
// that share their K/V tiles; warps 2-5 run one tile's online softmax and
// warps 6-9 the other's, one thread per query row, while the MMA thread
// interleaves the two tiles' Q K^T and P V. P is written back over its S
// columns as packed bf16 and read from TMEM as the A operand of O += P V; O
// is rescaled in place only when a row maximum grows by more than 2^8. The
// log-sum-exp of every row is saved.
//
// Backward (head_dim 64 or 128) in two kernels, so no dQ atomics are needed
// and the result does not depend on scheduling:
//  * dK/dV, one CTA per (128-key tile, kv head, sequence), loops over the
//    query heads of its group and the 64-query tiles at or below the
//    diagonal (Q, dO and their lse / D rows through a 4-deep ring, so the
//    copies run well ahead of the two TMEM buffer pairs): S^T = K Q^T and dP^T = V dO^T into one of two TMEM buffer
//    pairs; P^T and dS^T = P^T o (dP^T - D) are written back over their own
//    TMEM columns as packed bf16 and read as the A operands of dV += P^T dO
//    and dK += dS^T Q, which accumulate in TMEM over the whole group (the
//    GQA reduction costs nothing);
//  * dQ, persistent: each CTA walks (128-query tile, head, sequence) items
//    longest first; S and dP are recomputed per key tile, dS is written to
//    TMEM as packed bf16 (two buffers) and read as the A operand of
//    dQ += dS K, which accumulates in TMEM and is written once per item
//    while the next item's first scores are computed; K comes through a
//    3-deep ring (it is read again by dQ += dS K after the elementwise
//    pass), V through a 2-deep one freed as soon as dP = dO V^T completes;
//    both rings run across items.
// Every operand transposition is a shared-memory descriptor, never a copy.
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace rdt {

namespace {
constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kLn2F = 0.6931471805599453f;
constexpr int kThreads = 320;
constexpr int kEltThreads = 256;  // warps 2-9
}  // namespace

// Store 32 fp32 values (scaled) as fp32 or bf16 row segments.
__device__ __forceinline__ void store_row32_f32(float* dst, const uint32_t (&a)[32], float sc) {
#pragma unroll
  for (int e = 0; e < 8; ++e)
    reinterpret_cast<float4*>(dst)[e] =
        make_float4(__uint_as_float(a[4 * e]) * sc, __uint_as_float(a[4 * e + 1]) * sc,
                    __uint_as_float(a[4 * e + 2]) * sc, __uint_as_float(a[4 * e + 3]) * sc);
}
__device__ __forceinline__ void store_row32_bf16(bf16* dst, const uint32_t (&a)[32], float sc) {
#pragma unroll
  for (int e = 0; e < 4; ++e)
    reinterpret_cast<uint4*>(dst)[e] = make_uint4(
        pack_bf16x2(__uint_as_float(a[8 * e]) * sc, __uint_as_float(a[8 * e + 1]) * sc),
        pack_bf16x2(__uint_as_float(a[8 * e + 2]) * sc, __uint_as_float(a[8 * e + 3]) * sc),
        pack_bf16x2(__uint_as_float(a[8 * e + 4]) * sc, __uint_as_float(a[8 * e + 5]) * sc),
        pack_bf16x2(__uint_as_float(a[8 * e + 6]) * sc, __uint_as_float(a[8 * e + 7]) * sc));
}

// ============================================================== forward
// Rows rescale O only when their running maximum grows by more than 2^8 (in
// the log2 domain): below that the stale maximum is kept, P stays <= 2^8 and
// the result is the same (O and l are both relative to the stale maximum).
constexpr float kRescaleLog2 = 8.f;

// ---------------------------------------------------- forward, two tiles
// Each work item is a pair of 128-query tiles (A: queries [256 i, 256 i + 128),
// B: the next 128) of one query head and sequence; both read the same K/V
// tiles. Warps 2-5 run the online softmax of tile A and warps 6-9 that of
// tile B, one thread per query row (whole rows: no cross-warp reduction).
// The MMA thread interleaves the two tiles,
//   S_A(0) S_B(0) | PV_A(0) S_A(1) | PV_B(0) S_B(1) | PV_A(1) S_A(2) | ...
// so one tile's scores and P V run on the tensor cores while the other tile's
// softmax runs. Each tile has one S buffer in TMEM (P is written back over it
// as packed bf16 and read as the A operand of P V; tcgen05 operations of one
// thread complete in order, so S(j+1) issued after P V(j) cannot overwrite P
// early) and one O buffer, read out by its softmax group after the item's
// last P V. K and V tiles come through rings freed by tile B's S and P V.
template <int D>
struct Fwd2Cfg {
  static constexpr int BM = 128, BN = 128;
  static constexpr uint32_t CHUNK = 128 * 128;  // 64 cols x 128 rows of bf16
  static constexpr uint32_t Q_BYTES = BM * D * 2;
  static constexpr uint32_t KV_BYTES = BN * D * 2;
  static constexpr int KS = D == 128 ? 2 : 3;
  static constexpr int VS = D == 128 ? 2 : 3;
  static constexpr uint32_t OFF_Q = 0;                       // [2]: tiles A, B
  static constexpr uint32_t OFF_K = OFF_Q + 2 * Q_BYTES;     // [KS]
  static constexpr uint32_t OFF_V = OFF_K + KS * KV_BYTES;   // [VS]
  static constexpr uint32_t OFF_BAR = OFF_V + VS * KV_BYTES;
  static constexpr size_t SMEM = OFF_BAR + 512 + 1024;
  // TMEM: S_A, S_B (128 fp32 columns each), then O_A, O_B (D columns each)
  static constexpr uint32_t TMEM_S = 0, TMEM_O = 256, TMEM_COLS = 512;
  static_assert(TMEM_O + 2 * D <= TMEM_COLS, "two O buffers must fit in TMEM");
  static_assert(SMEM <= 232448, "attention forward tile exceeds the shared memory of a CTA");
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd2_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, bf16* __restrict__ o,
                     float* __restrict__ lse, int B, int S, int nh, int nkv, float scale_log2,
                     int* err) {
  using C = Fwd2Cfg<D>;
  constexpr int BM = C::BM, BN = C::BN, DCH = D / 64, KS = C::KS, VS = C::VS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  // barriers: q_full, q_empty, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS],
  // s_full[2], p_full[2], o_done[2], o_free[2], drain
  const uint32_t q_full = bar0, q_empty = bar0 + 8, k_full = bar0 + 16,
                 k_empty = k_full + 8 * KS, v_full = k_empty + 8 * KS, v_empty = v_full + 8 * VS,
                 s_full = v_empty + 8 * VS, p_full = s_full + 16, o_done = p_full + 16,
                 o_free = o_done + 16, drain = o_free + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 384);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qp = (S + 2 * BM - 1) / (2 * BM);
  const int n_kvt = (S + BN - 1) / BN;
  const int per = nh * B;
  const int n_items = n_qp * per;
  const int grp = nh / nkv;
  // item idx -> pair i (longest first), head h, sequence b; tiles of A and B
  auto item = [&](int idx, int& i, int& h, int& b, int& nA, int& nB) {
    i = n_qp - 1 - idx / per;
    const int rem = idx % per;
    h = rem % nh;
    b = rem / nh;
    nA = min(2 * i + 1, n_kvt);
    nB = min(2 * i + 2, n_kvt);
  };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int x = 0; x < KS; ++x) {
      mbar_init(k_full + 8 * x, 1);
      mbar_init(k_empty + 8 * x, 1);
    }
    for (int x = 0; x < VS; ++x) {
      mbar_init(v_full + 8 * x, 1);
      mbar_init(v_empty + 8 * x, 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(s_full + 8 * x, 1);
      mbar_init(p_full + 8 * x, 128);
      mbar_init(o_done + 8 * x, 1);
      mbar_init(o_free + 8 * x, 128);
    }
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
      bool ok = true;
      int jg = 0;
      for (int idx = blockIdx.x, it = 0; idx < n_items && ok; idx += gridDim.x, ++it) {
        int i, h, b, nA, nB;
        item(idx, i, h, b, nA, nB);
        const int g = h / grp, tok0 = b * S;
        if (!mbar_wait(q_empty, (it & 1) ^ 1, err)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(q_full, 2 * C::Q_BYTES);
        for (int x = 0; x < 2; ++x)
          for (int c = 0; c < DCH; ++c)
            tma_load_2d(sbase + C::OFF_Q + x * C::Q_BYTES + c * C::CHUNK, &tq, q_full,
                        h * D + c * 64, tok0 + 2 * BM * i + BM * x);
        auto load_k = [&](int j) -> bool {
          const int jj = jg + j, st = jj % KS;
          if (!mbar_wait(k_empty + 8 * st, ((jj / KS) & 1) ^ 1, err)) return false;
          mbar_arrive_expect_tx(k_full + 8 * st, C::KV_BYTES);
          for (int c = 0; c < DCH; ++c)
            tma_load_2d(sbase + C::OFF_K + st * C::KV_BYTES + c * C::CHUNK, &tk, k_full + 8 * st,
                        g * D + c * 64, tok0 + j * BN);
          return true;
        };
        auto load_v = [&](int j) -> bool {
          const int jj = jg + j, st = jj % VS;
          if (!mbar_wait(v_empty + 8 * st, ((jj / VS) & 1) ^ 1, err)) return false;
          mbar_arrive_expect_tx(v_full + 8 * st, C::KV_BYTES);
          for (int c = 0; c < DCH; ++c)
            tma_load_2d(sbase + C::OFF_V + st * C::KV_BYTES + c * C::CHUNK, &tv, v_full + 8 * st,
                        g * D + c * 64, tok0 + j * BN);
          return true;
        };
        for (int j = 0; j < KS - 1 && j < nB && ok; ++j) ok = load_k(j);
        for (int j = 0; j < nB && ok; ++j) {
          if (j + KS - 1 < nB) ok = load_k(j + KS - 1);
          if (ok) ok = load_v(j);
        }
        jg += nB;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------------------- MMA
      constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(BM, D, 0, 1);
      bool ok = true;
      int jg = 0, jt0 = 0, jt1 = 0;  // KV tiles so far; P V issued so far per tile
      for (int idx = blockIdx.x, it = 0; idx < n_items && ok; idx += gridDim.x, ++it) {
        int i, h, b, nA, nB;
        item(idx, i, h, b, nA, nB);
        // S_x(j) = Q_x K_j^T into tile x's S buffer
        auto issue_s = [&](int x, int j) -> bool {
          const int jj = jg + j, ks = jj % KS;
          if (!mbar_wait(k_full + 8 * ks, (jj / KS) & 1, err)) return false;
          tc_fence_after();
          const uint32_t kb = sbase + C::OFF_K + ks * C::KV_BYTES;
          const uint32_t qb = sbase + C::OFF_Q + x * C::Q_BYTES;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * C::CHUNK + (k & 3) * 32;
            tc_mma_bf16(tmem + C::TMEM_S + x * BN, sdesc_sw128(qb + off, 16, 1024),
                        sdesc_sw128(kb + off, 16, 1024), idesc_s, k > 0);
          }
          tc_commit(s_full + 8 * x);
          return true;
        };
        // O_x += P_x(j) V_j with P (bf16, over tile x's S buffer) from TMEM
        auto issue_pv = [&](int x, int j) -> bool {
          const int jj = jg + j, vs = jj % VS;
          if (j == 0 && !mbar_wait(o_free + 8 * x, (it & 1) ^ 1, err)) return false;
          if (!mbar_wait(p_full + 8 * x, (x ? jt1 : jt0) & 1, err) ||
              !mbar_wait(v_full + 8 * vs, (jj / VS) & 1, err))
            return false;
          tc_fence_after();
          const uint32_t vb = sbase + C::OFF_V + vs * C::KV_BYTES;
#pragma unroll
          for (int k = 0; k < BN / 16; ++k)
            tc_mma_bf16_ts(tmem + C::TMEM_O + x * D, tmem + C::TMEM_S + x * BN + k * 8,
                           sdesc_sw128(vb + k * 2048, C::CHUNK, 1024), idesc_o, (j | k) != 0);
          tc_commit(o_done + 8 * x);
          if (x) ++jt1;
          else ++jt0;
          return true;
        };
        if (!mbar_wait(q_full, it & 1, err)) {
          ok = false;
          break;
        }
        ok = issue_s(0, 0) && issue_s(1, 0);
        if (!ok) break;
        tc_commit(k_empty + 8 * (jg % KS));
        if (nB == 1) tc_commit(q_empty);
        for (int j = 0; j < nB && ok; ++j) {
          if (j < nA) {
            ok = issue_pv(0, j) && (j + 1 >= nA || issue_s(0, j + 1));
            if (!ok) break;
          }
          ok = issue_pv(1, j);
          if (!ok) break;
          tc_commit(v_empty + 8 * ((jg + j) % VS));
          if (j + 1 < nB) {
            ok = issue_s(1, j + 1);
            if (!ok) break;
            tc_commit(k_empty + 8 * ((jg + j + 1) % KS));
            if (j + 2 == nB) tc_commit(q_empty);  // the item's last Q K^T
          }
        }
        jg += nB;
      }
      tc_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else {
    // ------------------------------- softmax: one query row per thread
    const int x = (warp - 2) >> 2;  // 0: tile A, 1: tile B
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t ts = tmem + lane_base + C::TMEM_S + x * BN;
    const uint32_t t_o = tmem + lane_base + C::TMEM_O + x * D;
    bool ok = true;
    int jx = 0;  // tiles of this softmax group so far
    for (int idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x) {
      int i, h, b, nA, nB;
      item(idx, i, h, b, nA, nB);
      const int n_tiles = x ? nB : nA;
      const int qpos = 2 * BM * i + BM * x + row;
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < n_tiles; ++j, ++jx) {
        if (!warp_wait(s_full + 8 * x, jx & 1, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sv[128];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(ts + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32 * c]));
        tmem_ld_wait();
        // keys j BN + c with c < lim are visible to this row (causal, and
        // inside the sequence): only tiles on or past the diagonal mask
        const int lim = min(qpos + 1, S) - j * BN;
        if (__any_sync(0xffffffffu, lim < BN)) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= lim) sv[c] = __float_as_uint(-INFINITY);
        }
        // row maximum of the raw scores (the scale is positive), four chains
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < 128; ++c) m4[c & 3] = fmaxf(m4[c & 3], __uint_as_float(sv[c]));
        const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * scale_log2;
        float alpha = 1.f;
        if (mx > m_run + kRescaleLog2) {
          alpha = (m_run == -INFINITY) ? 0.f : ex2_approx(m_run - mx);
          m_run = mx;
        }
        // p = 2^(s scale - m), one FMA per score; bf16 pairs in place
        const float nm = -m_run;
        float s2[2] = {0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(sv[c]), scale_log2, nm));
          const float p1 = ex2_approx(fmaf(__uint_as_float(sv[c + 1]), scale_log2, nm));
          s2[(c >> 1) & 1] += p0 + p1;
          sv[c / 2] = pack_bf16x2(p0, p1);
        }
        l_run = l_run * alpha + (s2[0] + s2[1]);
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // O is being accumulated by P V of the previous tile until it completes
          if (!warp_wait(o_done + 8 * x, (jx - 1) & 1, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(t_o + c * 32, ov);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st32(t_o + c * 32, ov);
          }
        }
        // P: 128 keys as 64 bf16 pairs over the first 64 columns of S
        tmem_st32(ts, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tmem_st32(ts + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_full + 8 * x);
      }
      if (!ok || !warp_wait(o_done + 8 * x, (jx - 1) & 1, err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      bf16* orow = o + (int64_t)(b * S + qpos) * (nh * D) + h * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(t_o + c * 32, ov);
        tmem_ld_wait();
        if (qpos < S) store_row32_bf16(orow + c * 32, ov, inv);
      }
      // this O buffer is free for the next item
      tc_fence_before();
      mbar_arrive(o_free + 8 * x);
      if (qpos < S) lse[((int64_t)b * nh + h) * S + qpos] = (m_run + __log2f(l_run)) * kLn2F;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (err && *reinterpret_cast<volatile int*>(err) != 0) {
    // after a timed-out wait, copies issued just before may still be landing
    // in this CTA's shared memory: let them finish before it exits
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 200000ull) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ============================================================= backward
// The log2-domain LSE and D = rowsum(dO o O) are read from [B*nh, S_pad]
// arrays (S_pad a multiple of 64) so that 64-query segments are aligned.
template <int D_>
struct BwdCfg {
  static constexpr int D = D_, BKV = 128, BQ = 64;
  static constexpr uint32_t KV_CHUNK = 128 * 128;  // 64 d-cols x 128 key rows
  static constexpr uint32_t Q_CHUNK = 64 * 128;    // 64 d-cols x 64 query rows
  static constexpr uint32_t KV_BYTES = BKV * D * 2;
  static constexpr uint32_t Q_BYTES = BQ * D * 2;
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + KV_BYTES;
  // Q / dO / (lse, D) stages: the loads for query tile it + 2 wait for dV/dK
  // of tile it - QST + 2 to free their stage, so with QST = 4 their latency
  // stays off the path S -> P -> dV/dK that the two TMEM buffer pairs allow
  static constexpr int QST = 4;
  static constexpr uint32_t OFF_Q = OFF_V + KV_BYTES;        // [QST]
  static constexpr uint32_t OFF_DO = OFF_Q + QST * Q_BYTES;  // [QST]
  static constexpr uint32_t OFF_LD = OFF_DO + QST * Q_BYTES;  // float [QST][lse2, D][64]
  static constexpr uint32_t OFF_BAR = OFF_LD + QST * 2 * 64 * 4;
  static constexpr size_t SMEM = OFF_BAR + 256 + 1024;
  // TMEM columns: dK, dV, then two (S^T, dP^T) buffer pairs of 64 + 64
  // columns; P^T and dS^T (packed bf16) are written back over their own S^T /
  // dP^T columns and read from there as the A operands of dV += P^T dO and
  // dK += dS^T Q.
  static constexpr uint32_t T_DK = 0, T_DV = 128, T_S = 256;
  static constexpr uint32_t TMEM_COLS = 512;
};
static_assert(BwdCfg<128>::SMEM <= 232448, "dK/dV stages exceed the shared memory of a CTA");

// TMEM column (relative to an S^T / dP^T block) of the packed bf16 A operand
// for K step kk (16 queries): the lanes of warp half h pack their 32 queries
// into columns [32 h, 32 h + 16).
__device__ __forceinline__ uint32_t packed_kstep_col(int kk) {
  return static_cast<uint32_t>((kk >> 1) * 32 + (kk & 1) * 8);
}

template <int DH>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tq,
                            const __grid_constant__ CUtensorMap tk,
                            const __grid_constant__ CUtensorMap tv,
                            const __grid_constant__ CUtensorMap tdo,
                            const float* __restrict__ lse2, const float* __restrict__ Dd,
                            int S_pad, float* __restrict__ dk, bf16* __restrict__ dv,
                            int64_t lddv, int B, int S, int nh, int nkv, float scale,
                            float scale_log2, int* err) {
  using C = BwdCfg<DH>;
  constexpr int D = C::D, BKV = C::BKV, BQ = C::BQ, DCH = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  constexpr int QST = C::QST;
  // bars: kv_full, q_full[QST], q_empty[QST], s_full[2], p_ready[2], done[2], fin, drain
  const uint32_t kv_full = bar0, q_full = bar0 + 8, q_empty = q_full + 8 * QST,
                 s_full = q_empty + 8 * QST, p_ready = s_full + 16, done = p_ready + 16,
                 fin = done + 16, drain = fin + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 192);
  static_assert(8 * (4 + 2 * QST + 6) <= 192, "dK/dV barriers overlap the TMEM slot");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per = nkv * B;
  const int nt = static_cast<int>(blockIdx.x) / per;  // key tile 0 (most work) first
  const int g = (static_cast<int>(blockIdx.x) % per) % nkv;
  const int b = (static_cast<int>(blockIdx.x) % per) / nkv;
  const int rep = nh / nkv;
  const int n0 = nt * BKV;
  const int tok0 = b * S;
  const int q_tiles = (S + BQ - 1) / BQ;
  const int first_qt = n0 / BQ;
  const int per_head = q_tiles - first_qt;
  const int iters = rep * per_head;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < QST; ++i) {
      mbar_init(q_full + 8 * i, 1);
      mbar_init(q_empty + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + 8 * i, 1);
      mbar_init(p_ready + 8 * i, kEltThreads);
      mbar_init(done + 8 * i, 1);
    }
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
      for (int c = 0; c < DCH; ++c) {
        tma_load_2d(sbase + C::OFF_K + c * C::KV_CHUNK, &tk, kv_full, g * D + c * 64, tok0 + n0);
        tma_load_2d(sbase + C::OFF_V + c * C::KV_CHUNK, &tv, kv_full, g * D + c * 64, tok0 + n0);
      }
      uint32_t pending = 0;
      bool ok = true;
      for (int it = 0; it < iters && ok; ++it) {
        const int qs = it % QST;
        const uint32_t ph = (it / QST) & 1;
        if (!mbar_wait(q_empty + 8 * qs, ph ^ 1, err)) {
          ok = false;
          break;
        }
        const int hh = g * rep + it / per_head;
        const int m0 = (first_qt + it % per_head) * BQ;
        const uint32_t qf = q_full + 8 * qs;
        mbar_arrive_expect_tx(qf, 2 * C::Q_BYTES + 512);
        for (int c = 0; c < DCH; ++c) {
          tma_load_2d(sbase + C::OFF_Q + qs * C::Q_BYTES + c * C::Q_CHUNK, &tq, qf,
                      hh * D + c * 64, tok0 + m0);
          tma_load_2d(sbase + C::OFF_DO + qs * C::Q_BYTES + c * C::Q_CHUNK, &tdo, qf,
                      hh * D + c * 64, tok0 + m0);
        }
        const int64_t seg = ((int64_t)b * nh + hh) * S_pad + m0;
        bulk_load_1d(sbase + C::OFF_LD + qs * 512, lse2 + seg, 256, qf);
        bulk_load_1d(sbase + C::OFF_LD + qs * 512 + 256, Dd + seg, 256, qf);
        pending = (pending & ~(3u << (2 * qs))) | ((1u | (ph << 1)) << (2 * qs));
      }
      if (!ok) {
        mbar_wait(kv_full, 0, nullptr);
        for (int qs = 0; qs < QST; ++qs)
          if ((pending >> (2 * qs)) & 1u)
            mbar_wait(q_full + 8 * qs, (pending >> (2 * qs + 1)) & 1u, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------------------- MMA
      constexpr uint32_t id_s = idesc_bf16_f32(128, BQ, 0, 0);  // S^T, dP^T
      constexpr uint32_t id_kv = idesc_bf16_f32(128, D, 0, 1);  // dV, dK (A from TMEM)
      const uint64_t k_desc = sdesc_sw128(sbase + C::OFF_K, 16, 1024);
      const uint64_t v_desc = sdesc_sw128(sbase + C::OFF_V, 16, 1024);
      bool ok = mbar_wait(kv_full, 0, err);
      auto issue_s = [&](int it) -> bool {
        const int st = it & 1, qs = it % QST;
        if (!mbar_wait(q_full + 8 * qs, (it / QST) & 1, err)) return false;
        // buffer pair st still holds P^T / dS^T of iteration it - 2
        if (it >= 2 && !mbar_wait(done + 8 * st, ((it >> 1) & 1) ^ 1, err)) return false;
        tc_fence_after();
        const uint64_t q_desc = sdesc_sw128(sbase + C::OFF_Q + qs * C::Q_BYTES, 16, 1024);
        const uint64_t o_desc = sdesc_sw128(sbase + C::OFF_DO + qs * C::Q_BYTES, 16, 1024);
        const uint32_t ts = tmem + C::T_S + st * 128;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t kv_off = ((k >> 2) * C::KV_CHUNK + (k & 3) * 32) >> 4;
          const uint64_t q_off = ((k >> 2) * C::Q_CHUNK + (k & 3) * 32) >> 4;
          tc_mma_bf16(ts, k_desc + kv_off, q_desc + q_off, id_s, k > 0);
          tc_mma_bf16(ts + 64, v_desc + kv_off, o_desc + q_off, id_s, k > 0);
        }
        tc_commit(s_full + 8 * st);
        return true;
      };
      if (ok && iters > 0) ok = issue_s(0);
      for (int it = 0; it < iters && ok; ++it) {
        const int st = it & 1;
        if (it + 1 < iters && !issue_s(it + 1)) {
          ok = false;
          break;
        }
        if (!mbar_wait(p_ready + 8 * st, (it >> 1) & 1, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int qs = it % QST;
        const uint32_t qb = sbase + C::OFF_Q + qs * C::Q_BYTES;
        const uint32_t ob = sbase + C::OFF_DO + qs * C::Q_BYTES;
        const uint32_t ts = tmem + C::T_S + st * 128;
#pragma unroll
        for (int k = 0; k < BQ / 16; ++k) {
          // dV += P^T dO ; dK += dS^T Q   (K dimension = query rows)
          tc_mma_bf16_ts(tmem + C::T_DV, ts + packed_kstep_col(k),
                         sdesc_sw128(ob + k * 2048, C::Q_CHUNK, 1024), id_kv, (it | k) != 0);
          tc_mma_bf16_ts(tmem + C::T_DK, ts + 64 + packed_kstep_col(k),
                         sdesc_sw128(qb + k * 2048, C::Q_CHUNK, 1024), id_kv, (it | k) != 0);
        }
        tc_commit(done + 8 * st);
        tc_commit(q_empty + 8 * qs);
      }
      tc_commit(fin);
      tc_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else {
    // ------------------- P^T and dS^T (key row, 32 of the 64 query columns)
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;  // key row within the tile
    const int kpos = n0 + row;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = true;
    for (int it = 0; it < iters; ++it) {
      const int st = it & 1;
      const int m0 = (first_qt + it % per_head) * BQ;
      if (!warp_wait(s_full + 8 * st, (it >> 1) & 1, err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[32], dp[32];
      const uint32_t ts = tmem + lane_base + C::T_S + st * 128 + half * 32;
      tmem_ld32(ts, sv);
      tmem_ld32(ts + 64, dp);
      tmem_ld_wait();
      const int qs = it % QST;
      const float4* l4 = reinterpret_cast<const float4*>(smem + C::OFF_LD + qs * 512) + half * 8;
      const float4* d4 =
          reinterpret_cast<const float4*>(smem + C::OFF_LD + qs * 512 + 256) + half * 8;
      const int q0 = m0 + half * 32;
      // queries q0 + c with lo <= c < hi see this key row (causal, inside the
      // sequence); the mask is applied only where some row of the warp needs it
      const int lo = kpos - q0, hi = kpos < S ? S - q0 : 0;
      const bool full = __all_sync(0xffffffffu, lo <= 0 && hi >= 32);
      // bf16 pairs of P^T / dS^T are packed in place into sv / dp [0, 16)
      auto pass = [&](auto masked) {
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 lv = l4[c4], dv4 = d4[c4];
          const float la[4] = {lv.x, lv.y, lv.z, lv.w}, da[4] = {dv4.x, dv4.y, dv4.z, dv4.w};
          float pv[4], dsv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = 4 * c4 + e;
            const float x = __uint_as_float(sv[c]) * scale_log2 - la[e];
            float p;
            if constexpr (decltype(masked)::value)
              p = (c >= lo && c < hi) ? ex2_approx(x) : 0.f;
            else
              p = ex2_approx(x);
            pv[e] = p;
            dsv[e] = p * (__uint_as_float(dp[c]) - da[e]);
          }
          sv[2 * c4] = pack_bf16x2(pv[0], pv[1]);
          sv[2 * c4 + 1] = pack_bf16x2(pv[2], pv[3]);
          dp[2 * c4] = pack_bf16x2(dsv[0], dsv[1]);
          dp[2 * c4 + 1] = pack_bf16x2(dsv[2], dsv[3]);
        }
      };
      if (full)
        pass(std::false_type{});
      else
        pass(std::true_type{});
      // over this warp's own S^T / dP^T columns (no other warp reads them)
      tmem_st16(ts, *reinterpret_cast<uint32_t(*)[16]>(&sv[0]));
      tmem_st16(ts + 64, *reinterpret_cast<uint32_t(*)[16]>(&dp[0]));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_ready + 8 * st);
    }
    // dK (scaled) and dV of this key tile, summed over the query heads of the group
    if (ok && warp_wait(fin, 0, err)) {
      tc_fence_after();
      float* dkr = dk + (int64_t)(tok0 + kpos) * (nkv * D) + g * D + half * (D / 2);
      bf16* dvr = dv + (int64_t)(tok0 + kpos) * lddv + g * D + half * (D / 2);
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t a[32], v[32];
        tmem_ld32(tmem + lane_base + C::T_DK + half * (D / 2) + c * 32, a);
        tmem_ld32(tmem + lane_base + C::T_DV + half * (D / 2) + c * 32, v);
        tmem_ld_wait();
        if (kpos < S) {
          store_row32_f32(dkr + c * 32, a, scale);
          store_row32_bf16(dvr + c * 32, v, 1.0f);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// dQ (query-stationary): per (128-query tile, head, sequence) the scores and
// dP are recomputed for every 128-key tile at or below the diagonal and
// dQ += dS K accumulates in TMEM, so dQ is written once with plain stores.
template <int D_>
struct DqCfg {
  static constexpr int D = D_, BM = 128, BN = 128;
  static constexpr uint32_t CHUNK = 128 * 128;  // 64 cols x 128 rows of bf16
  static constexpr uint32_t T_BYTES = 128 * D * 2;
  // K runs three tiles deep (it is read by S = Q K^T and again, a whole
  // elementwise pass later, by dQ += dS K); V two (only dP = dO V^T reads it)
  static constexpr int KST = 3, VST = 2;
  static constexpr uint32_t OFF_Q = 0, OFF_DO = T_BYTES, OFF_K = 2 * T_BYTES,  // K[KST]
      OFF_V = OFF_K + KST * T_BYTES,                                             // V[VST]
      OFF_BAR = OFF_V + VST * T_BYTES;
  static constexpr size_t SMEM = OFF_BAR + 256 + 1024;
  // TMEM: S, dP (128 fp32 columns each), dQ (D columns), then two dS buffers
  // of 64 columns (128 keys as packed bf16 pairs, key 2i and 2i + 1 in
  // column i), the A operand of dQ += dS K.
  static constexpr uint32_t T_S = 0, T_DP = 128, T_DQ = 256, T_DS = 384, TMEM_COLS = 512;
};
static_assert(DqCfg<128>::SMEM <= 232448, "dQ stages exceed the shared memory of a CTA");

template <int DH>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                          const __grid_constant__ CUtensorMap tv,
                          const __grid_constant__ CUtensorMap tdo, const float* __restrict__ lse2,
                          const float* __restrict__ Dd, int S_pad, float* __restrict__ dq, int B,
                          int S, int nh, int nkv, float scale, float scale_log2, int* err) {
  using C = DqCfg<DH>;
  constexpr int D = C::D, BM = C::BM, BN = C::BN, DCH = D / 64, KST = C::KST, VST = C::VST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  // bars: q_full, q_empty, k_full[3], k_empty[3], v_full[2], v_empty[2], s_full,
  // s_used, ds_ready, ds_free[2], dq_done, dq_free, drain
  const uint32_t q_full = bar0, q_empty = bar0 + 8, k_full = bar0 + 16,
                 k_empty = k_full + 8 * KST, v_full = k_empty + 8 * KST,
                 v_empty = v_full + 8 * VST, s_full = v_empty + 8 * VST, s_used = s_full + 8,
                 ds_ready = s_used + 8, ds_free = ds_ready + 8, dq_done = ds_free + 16,
                 dq_free = dq_done + 8, drain = dq_free + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 192);
  static_assert(8 * (2 + 2 * KST + 2 * VST + 8) <= 192, "dQ barriers overlap the TMEM slot");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qt = (S + BM - 1) / BM;
  const int per = nh * B;
  const int n_items = n_qt * per;
  const int grp = nh / nkv;
  // item idx (longest rows first) -> query tile mt, head h, sequence b
  auto item = [&](int idx, int& mt, int& h, int& b) {
    mt = n_qt - 1 - idx / per;
    const int rem = idx % per;
    h = rem % nh;
    b = rem / nh;
  };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < KST; ++i) {
      mbar_init(k_full + 8 * i, 1);
      mbar_init(k_empty + 8 * i, 1);
    }
    for (int i = 0; i < VST; ++i) {
      mbar_init(v_full + 8 * i, 1);
      mbar_init(v_empty + 8 * i, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_used, kEltThreads);
    mbar_init(ds_ready, kEltThreads);
    mbar_init(ds_free, 1);
    mbar_init(ds_free + 8, 1);
    mbar_init(dq_done, 1);
    mbar_init(dq_free, kEltThreads);
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
      bool ok = true;
      int jg = 0;  // key tiles loaded so far (the rings run across items)
      for (int idx = blockIdx.x, it = 0; idx < n_items && ok; idx += gridDim.x, ++it) {
        int mt, h, b;
        item(idx, mt, h, b);
        const int g = h / grp, tok0 = b * S, n_tiles = min(n_qt, mt + 1);
        // Q and dO of this item once the previous item's last S / dP have read theirs
        if (!mbar_wait(q_empty, (it & 1) ^ 1, err)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(q_full, 2 * C::T_BYTES);
        for (int c = 0; c < DCH; ++c) {
          tma_load_2d(sbase + C::OFF_Q + c * C::CHUNK, &tq, q_full, h * D + c * 64,
                      tok0 + mt * BM);
          tma_load_2d(sbase + C::OFF_DO + c * C::CHUNK, &tdo, q_full, h * D + c * 64,
                      tok0 + mt * BM);
        }
        for (int j = 0; j < n_tiles && ok; ++j) {
          const int jj = jg + j, ks = jj % KST, vs = jj % VST;
          if (!mbar_wait(k_empty + 8 * ks, ((jj / KST) & 1) ^ 1, err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(k_full + 8 * ks, C::T_BYTES);
          for (int c = 0; c < DCH; ++c)
            tma_load_2d(sbase + C::OFF_K + ks * C::T_BYTES + c * C::CHUNK, &tk, k_full + 8 * ks,
                        g * D + c * 64, tok0 + j * BN);
          if (!mbar_wait(v_empty + 8 * vs, ((jj / VST) & 1) ^ 1, err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(v_full + 8 * vs, C::T_BYTES);
          for (int c = 0; c < DCH; ++c)
            tma_load_2d(sbase + C::OFF_V + vs * C::T_BYTES + c * C::CHUNK, &tv, v_full + 8 * vs,
                        g * D + c * 64, tok0 + j * BN);
        }
        jg += n_tiles;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------------------- MMA
      constexpr uint32_t id_s = idesc_bf16_f32(BM, BN, 0, 0);  // S, dP
      constexpr uint32_t id_q = idesc_bf16_f32(BM, D, 0, 1);   // dQ (A = dS from TMEM)
      bool ok = true;
      int jg = 0;
      for (int idx = blockIdx.x, it = 0; idx < n_items && ok; idx += gridDim.x, ++it) {
        int mt, h, b;
        item(idx, mt, h, b);
        const int n_tiles = min(n_qt, mt + 1);
        // S = Q K^T and dP = dO V^T of key tile j, once the elementwise warps
        // have read the previous tile's S and dP
        auto issue_s = [&](int j) -> bool {
          const int jj = jg + j, ks = jj % KST, vs = jj % VST;
          if (!mbar_wait(k_full + 8 * ks, (jj / KST) & 1, err) ||
              !mbar_wait(v_full + 8 * vs, (jj / VST) & 1, err) ||
              !mbar_wait(s_used, (jj & 1) ^ 1, err))
            return false;
          tc_fence_after();
          const uint32_t kb = sbase + C::OFF_K + ks * C::T_BYTES;
          const uint32_t vb = sbase + C::OFF_V + vs * C::T_BYTES;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * C::CHUNK + (k & 3) * 32;
            tc_mma_bf16(tmem + C::T_S, sdesc_sw128(sbase + C::OFF_Q + off, 16, 1024),
                        sdesc_sw128(kb + off, 16, 1024), id_s, k > 0);
            tc_mma_bf16(tmem + C::T_DP, sdesc_sw128(sbase + C::OFF_DO + off, 16, 1024),
                        sdesc_sw128(vb + off, 16, 1024), id_s, k > 0);
          }
          tc_commit(s_full);
          tc_commit(v_empty + 8 * vs);  // V is read by dP only
          if (j + 1 == n_tiles) tc_commit(q_empty);  // the item's last read of Q and dO
          return true;
        };
        if (!mbar_wait(q_full, it & 1, err) || !issue_s(0)) {
          ok = false;
          break;
        }
        for (int j = 0; j < n_tiles && ok; ++j) {
          const int jj = jg + j, ks = jj % KST;
          if (j + 1 < n_tiles && !issue_s(j + 1)) {
            ok = false;
            break;
          }
          // dQ of the previous item has been read out of TMEM
          if (j == 0 && !mbar_wait(dq_free, (it & 1) ^ 1, err)) {
            ok = false;
            break;
          }
          if (!mbar_wait(ds_ready, jj & 1, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t kb = sbase + C::OFF_K + ks * C::T_BYTES;
          const uint32_t ds = tmem + C::T_DS + (jj & 1) * 64;
#pragma unroll
          for (int k = 0; k < BN / 16; ++k)
            tc_mma_bf16_ts(tmem + C::T_DQ, ds + 8 * k, sdesc_sw128(kb + k * 2048, C::CHUNK, 1024),
                           id_q, (j | k) != 0);
          tc_commit(ds_free + 8 * (jj & 1));
          tc_commit(k_empty + 8 * ks);
        }
        if (ok) tc_commit(dq_done);
        jg += n_tiles;
      }
      tc_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else {
    // ---------------------------- dS (query row, 64 of the 128 key columns)
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = true;
    int jg = 0;
    for (int idx = blockIdx.x, it = 0; idx < n_items && ok; idx += gridDim.x, ++it) {
      int mt, h, b;
      item(idx, mt, h, b);
      const int n_tiles = min(n_qt, mt + 1);
      const int qpos = mt * BM + row;
      const bool qvalid = qpos < S;
      const int64_t seg = ((int64_t)b * nh + h) * S_pad + qpos;
      const float l2 = qvalid ? lse2[seg] : 0.f;
      const float drow = qvalid ? Dd[seg] : 0.f;
      for (int j = 0; j < n_tiles; ++j) {
        const int jj = jg + j;
        if (!warp_wait(s_full, jj & 1, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int c0 = j * BN + half * 64;
        // keys c0 + c with c < lim are visible to this query row; the mask is
        // applied only where some row of the warp needs it (diagonal tiles)
        const int lim = qvalid ? qpos + 1 - c0 : 0;
        const bool full = __all_sync(0xffffffffu, lim >= 64);
        uint32_t pk[32];
#pragma unroll
        for (int qt = 0; qt < 2; ++qt) {
          uint32_t sv[32], dp[32];
          const uint32_t t0 = tmem + lane_base + half * 64 + qt * 32;
          tmem_ld32(t0 + C::T_S, sv);
          tmem_ld32(t0 + C::T_DP, dp);
          tmem_ld_wait();
          if (qt == 1) {
            // every S / dP column this thread reads is in registers: the next
            // tile's S and dP may overwrite them while this half is computed
            tc_fence_before();
            mbar_arrive(s_used);
          }
          if (full) {
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              float d2[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float p = ex2_approx(__uint_as_float(sv[c + e]) * scale_log2 - l2);
                d2[e] = p * (__uint_as_float(dp[c + e]) - drow);
              }
              pk[qt * 16 + c / 2] = pack_bf16x2(d2[0], d2[1]);
            }
          } else {
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              float d2[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float p = qt * 32 + c + e < lim
                                    ? ex2_approx(__uint_as_float(sv[c + e]) * scale_log2 - l2)
                                    : 0.f;
                d2[e] = p * (__uint_as_float(dp[c + e]) - drow);
              }
              pk[qt * 16 + c / 2] = pack_bf16x2(d2[0], d2[1]);
            }
          }
        }
        // dS buffer jj & 1 was last read by dQ += dS K of tile jj - 2
        if (!warp_wait(ds_free + 8 * (jj & 1), ((jj >> 1) & 1) ^ 1, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // keys c0 .. c0 + 63 as bf16 pairs: columns half * 32 .. + 31 of the buffer
        tmem_st32(tmem + lane_base + C::T_DS + (jj & 1) * 64 + half * 32, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(ds_ready);
      }
      jg += n_tiles;
      if (!ok || !warp_wait(dq_done, it & 1, err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float* out = dq + (int64_t)(b * S + qpos) * (nh * D) + h * D + half * (D / 2);
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t a[32];
        tmem_ld32(tmem + lane_base + C::T_DQ + half * (D / 2) + c * 32, a);
        tmem_ld_wait();
        if (qvalid) store_row32_f32(out + c * 32, a, scale);
      }
      // the dQ accumulator is free for the next item
      tc_fence_before();
      mbar_arrive(dq_free);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (err && *reinterpret_cast<volatile int*>(err) != 0) {
    // after a timed-out wait, copies issued just before may still be landing
    // in this CTA's shared memory: let them finish before it exits
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 200000ull) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ================================================================== host
int attn_lse_pad(int S) { return (S + 63) / 64 * 64; }

bool attn_tc_supported(int d, bool) { return d == 64 || d == 128; }

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
    cudaError_t e = cudaFuncSetAttribute(attn_fwd2_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Fwd2Cfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int n_qp = (S + 255) / 256;
  const float scale_log2 = kLog2eF / sqrtf((float)D);
  note_launch();
  const int n_items = n_qp * nh * B;
  const int grid = n_items < num_sms() ? n_items : num_sms();
  attn_fwd2_kernel<D><<<grid, kThreads, Fwd2Cfg<D>::SMEM, s>>>(
      tq, tk, tv, o, lse, B, S, nh, nkv, scale_log2, err);
  return cudaGetLastError();
}

cudaError_t attn_fwd_tc(const bf16* q, int64_t ldq, const bf16* k, int64_t ldk, const bf16* v,
                        int64_t ldv, bf16* o, float* lse, int B, int S, int nh, int nkv, int d,
                        int* err, cudaStream_t s) {
  if (d == 128) return fwd_tc_d<128>(q, ldq, k, ldk, v, ldv, o, lse, B, S, nh, nkv, err, s);
  if (d == 64) return fwd_tc_d<64>(q, ldq, k, ldk, v, ldv, o, lse, B, S, nh, nkv, err, s);
  return cudaErrorInvalidValue;
}

template <int D>
static cudaError_t bwd_tc_d(const bf16* q, int64_t ldq, const bf16* k, int64_t ldk, const bf16* v,
                            int64_t ldv, const bf16* dout, const float* lse2, const float* Dd,
                            float* dq, float* dk, bf16* dv, int64_t lddv, int B, int S, int nh,
                            int nkv, int* err, cudaStream_t s) {
  const int64_t T = (int64_t)B * S;
  CUtensorMap tq64, tdo64, tq128, tdo128, tk, tv;
  if (!make_tma_2d(&tq64, q, T, (int64_t)nh * D, ldq, 64) ||
      !make_tma_2d(&tdo64, dout, T, (int64_t)nh * D, (int64_t)nh * D, 64) ||
      !make_tma_2d(&tq128, q, T, (int64_t)nh * D, ldq, 128) ||
      !make_tma_2d(&tdo128, dout, T, (int64_t)nh * D, (int64_t)nh * D, 128) ||
      !make_tma_2d(&tk, k, T, (int64_t)nkv * D, ldk, 128) ||
      !make_tma_2d(&tv, v, T, (int64_t)nkv * D, ldv, 128))
    return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dkdv_tc_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)BwdCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_bwd_dq_tc_kernel<D>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DqCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const float scale = 1.0f / sqrtf((float)D);
  const int S_pad = attn_lse_pad(S);
  const int n_t = (S + 127) / 128;
  note_launch();
  attn_bwd_dkdv_tc_kernel<D><<<n_t * nkv * B, kThreads, BwdCfg<D>::SMEM, s>>>(
      tq64, tk, tv, tdo64, lse2, Dd, S_pad, dk, dv, lddv, B, S, nh, nkv, scale, scale * kLog2eF,
      err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  note_launch();
  const int dq_items = n_t * nh * B;  // persistent: one CTA per SM walks the items
  attn_bwd_dq_tc_kernel<D><<<dq_items < num_sms() ? dq_items : num_sms(), kThreads,
                             DqCfg<D>::SMEM, s>>>(tq128, tk, tv, tdo128, lse2, Dd, S_pad, dq, B,
                                                  S, nh, nkv, scale, scale * kLog2eF, err);
  return cudaGetLastError();
}

cudaError_t attn_bwd_tc(const bf16* q, int64_t ldq, const bf16* k, int64_t ldk, const bf16* v,
                        int64_t ldv, const bf16* dout, const float* lse2, const float* Dd,
                        float* dq, float* dk, bf16* dv, int64_t lddv, int B, int S, int nh,
                        int nkv, int d, int* err, cudaStream_t s) {
  if (d == 128)
    return bwd_tc_d<128>(q, ldq, k, ldk, v, ldv, dout, lse2, Dd, dq, dk, dv, lddv, B, S, nh, nkv,
                         err, s);
  if (d == 64)
    return bwd_tc_d<64>(q, ldq, k, ldk, v, ldv, dout, lse2, Dd, dq, dk, dv, lddv, B, S, nh, nkv,
                        err, s);
  return cudaErrorInvalidValue;
}

}  // namespace rdt
