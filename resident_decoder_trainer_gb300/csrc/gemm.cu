// Persistent tcgen05 BF16 GEMM for sm_103a with fused epilogues.
//
// Single-CTA kernel, one CTA per SM (320 threads, ~197 KB shared memory, all
// 512 TMEM columns):
//   warp 0  TMA producer: streams 128x64 A and BNx64 B tiles (BN = 256 or
//           192; 128-byte swizzle) into a 4- or 5-stage shared-memory ring,
//           one mbarrier per stage;
//   warp 1  MMA issuer: one elected lane issues tcgen05.mma (M=128, N=BN,
//           K=16) into one of two TMEM accumulators (2 x BN fp32 columns),
//           then tcgen05.commit frees the smem stage / signals the epilogue;
//   warps 2-9 epilogue: two warps per 32-lane TMEM quarter, each taking half of
//           the tile's columns; tcgen05.ld (one output row per thread), fused
//           elementwise work, vectorised global stores; the accumulator is
//           handed back so the next tile's MMAs overlap.
// CTA-pair kernel (gemm2_kernel, below): the same roles on clusters of two
// CTAs with 256 x 256 tiles and the pair MMA (cta_group::2).
// Operands may be K-major ([rows, K], K contiguous) or MN-major ([K, rows]);
// the transposed cases are expressed through the UMMA descriptors, so no
// operand is ever transposed in memory. Ragged M/N/K edges are zero-filled by
// TMA and masked in the epilogue.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace rdt {

constexpr int BM = 128, BK = 64;
constexpr uint32_t A_BYTES = BM * BK * 2;         // 16 KB
constexpr uint32_t MN_CHUNK_BYTES = 64 * BK * 2;  // one 64-row x 64-col box: 8 KB
constexpr int GEMM_THREADS = 320;
constexpr int EPI_THREADS = 256;
constexpr int TMEM_COLS = 512;

// Epilogue staging per epilogue warp (two buffers, see the epilogues below):
// 4 KB; 128 x 192 tiles keep a 5-stage ring by staging 2 KB per warp (in
// units half as wide).
__host__ __device__ constexpr uint32_t OutStageBytes(int bn) { return bn == 192 ? 2048 : 4096; }
template <int BN, bool PAIR>
struct OutStage {
  static constexpr uint32_t BYTES = OutStageBytes(BN);
  static constexpr uint32_t TOTAL = BYTES * (EPI_THREADS / 32);
};

// Tile width N = BN (256 or 192). Shared memory: a ring of 64-deep stages
// (4 of 48 KB or 5 of 40 KB), the epilogue's output staging (32 or 16 KB),
// barriers.
template <int BN_>
struct Tile {
  static constexpr int BN = BN_;
  static constexpr uint32_t B_BYTES = BN * BK * 2;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = BN == 256 ? 4 : 5;
  static constexpr uint32_t OFF_OUT = STAGES * STAGE_BYTES;
  static constexpr size_t SMEM = OFF_OUT + OutStage<BN, false>::TOTAL + 1024 + 512;
};

struct GemmParams {
  int M, N, K;
  int m_tiles, n_tiles, k_blocks;
  int swiglu_half;  // SwiGLU: row offset of the up rows in the stacked [2I, K] B
  int group;        // rasterisation: row tiles per group (see tile_coords)
  int sq_slots;     // squared-sum slots per tile (8 single-CTA, 16 pair)
  int kb_main;      // NF4 GEMM: k-blocks of the decoded operand; the rest are the tail
  // split-K (single-CTA kernel): work unit u is tile u % tiles over k-blocks
  // [s kb_split, (s + 1) kb_split) with s = u / tiles; its fp32 partial lands
  // in rows s m_pad + (tile rows) of the output. splits = 1: whole K.
  int splits, kb_split, m_pad;
  int m_epi;        // rows the epilogue may write (M, or splits m_pad)
  Epi epi;
  int* err;
};

// Tile t -> (row tile, column tile). Groups of p.group row tiles sweep all
// column tiles, row tile fastest. group = m_tiles keeps all of A resident in L2
// while B streams through once; group = 1 does the same for B (column tile
// fastest); the host picks the one whose resident operand fits in L2.
__device__ __forceinline__ void tile_coords(int t, const GemmParams& p, int& mt, int& nt) {
  const int G = p.group;
  const int per_group = G * p.n_tiles;
  const int g = t / per_group;
  const int first = g * G;
  const int gs = min(p.m_tiles - first, G);
  const int r = t - g * per_group;
  mt = first + r % gs;
  nt = r / gs;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

// -------------------------------------------------------------- epilogues
// Each epilogue warp owns 32 rows (its TMEM lane quarter) and half of the
// tile's columns, and streams them out in units of UNIT columns through two
// staging buffers (STG/2 bytes each) in shared memory:
//   * every thread writes its row of the unit into the buffer in the layout of
//     a TMA box with the matching swizzle (rows of 16, 32, 64 or 128 bytes;
//     conflict-free), and one lane writes the box with a bulk tensor store
//     (whole lines; the tensor map clips it at M and, in 16-byte units, N);
//   * the buffers alternate, so a unit is written while the previous unit's
//     store is still reading the other buffer;
//   * inputs of the residual and SwiGLU-backward epilogues arrive the same way
//     in reverse: a TMA load of the next unit's residual / g / u box is in
//     flight while the current unit is computed in place.
__host__ __device__ constexpr int epi_unit(int kind, uint32_t stg) {
  return kind == EPI_SWIGLU ? 32                                      // g+u, then s
         : (kind == EPI_BF16 || kind == EPI_CE || kind == EPI_CE_GRAD) ? (stg >= 4096 ? 32 : 16)
                                               : (stg >= 4096 ? 16 : 8);  // fp32; g+u in, dg+du out
}
__host__ __device__ constexpr int epi_elem_bytes(int kind) {
  return (kind == EPI_F32 || kind == EPI_F32_RESID) ? 4 : 2;
}

// Output / input tensor maps: o1 = out (g for SwiGLU, dg for SwiGLU-bwd,
// logits for CE), o2 = u / du, o3 = s; i1 = residual or g, i2 = u.
struct OutMaps {
  CUtensorMap o1, o2, o3, i1, i2;
};

struct Stage {
  uint8_t* p;    // this warp's two staging buffers
  uint32_t a;    // their shared-memory address
  uint32_t bar;  // this warp's two input mbarriers
  int lane;
};

// Offset of 16-byte chunk k of row r in a block of 32 rows x RB bytes, as a
// TMA box with 128/64/32-byte swizzle (RB = 128/64/32) or none (RB = 16).
template <uint32_t RB>
__device__ __forceinline__ uint32_t stg_off(int r, int k) {
  constexpr int sh = RB == 128 ? 0 : RB == 64 ? 1 : RB == 32 ? 2 : 3;
  constexpr int mask = static_cast<int>(RB / 16) - 1;
  return r * RB + static_cast<uint32_t>(((k ^ (r >> sh)) & mask) << 4);
}

// Row `lane` of a unit: UNIT fp32 values as fp32 or bf16.
template <uint32_t RB, int UNIT>
__device__ __forceinline__ void put_f32(uint8_t* b, int lane, const float* v) {
#pragma unroll
  for (int k = 0; k < UNIT / 4; ++k)
    *reinterpret_cast<float4*>(b + stg_off<RB>(lane, k)) =
        make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
}
template <uint32_t RB, int UNIT>
__device__ __forceinline__ void put_bf16(uint8_t* b, int lane, const float* v) {
#pragma unroll
  for (int k = 0; k < UNIT / 8; ++k)
    *reinterpret_cast<uint4*>(b + stg_off<RB>(lane, k)) =
        make_uint4(pack_bf16x2(v[8 * k], v[8 * k + 1]), pack_bf16x2(v[8 * k + 2], v[8 * k + 3]),
                   pack_bf16x2(v[8 * k + 4], v[8 * k + 5]),
                   pack_bf16x2(v[8 * k + 6], v[8 * k + 7]));
}
template <uint32_t RB, int UNIT>
__device__ __forceinline__ void get_f32(const uint8_t* b, int lane, float* v) {
#pragma unroll
  for (int k = 0; k < UNIT / 4; ++k) {
    const float4 q = *reinterpret_cast<const float4*>(b + stg_off<RB>(lane, k));
    v[4 * k] = q.x;
    v[4 * k + 1] = q.y;
    v[4 * k + 2] = q.z;
    v[4 * k + 3] = q.w;
  }
}
template <uint32_t RB, int UNIT>
__device__ __forceinline__ void get_bf16(const uint8_t* b, int lane, float* v) {
#pragma unroll
  for (int k = 0; k < UNIT / 8; ++k) {
    const uint4 q = *reinterpret_cast<const uint4*>(b + stg_off<RB>(lane, k));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      v[8 * k + 2 * h] = bf16lo(w[h]);
      v[8 * k + 2 * h + 1] = bf16hi(w[h]);
    }
  }
}

// One warp's share of a tile (rows row0 + [0, 32), half `half` of the
// columns). Waits for the accumulator itself (after starting the first input
// load); returns false if a bounded wait timed out. ucnt counts the warp's
// units over all its tiles (unit i uses buffer i & 1), eph holds the phase
// bit of each buffer's input barrier.
template <int EPI, int BN, uint32_t STG>
__device__ __forceinline__ bool epilogue_tile(const GemmParams& p, const OutMaps& om,
                                              uint32_t tbase, int row0, int nt, int half,
                                              const Stage& st, uint32_t& ucnt, uint32_t& eph,
                                              uint32_t tfull, uint32_t tfull_ph, int tile,
                                              int slot) {
  constexpr int UNIT = epi_unit(EPI, STG);
  constexpr uint32_t BUF = STG / 2;
  constexpr uint32_t RB = UNIT * epi_elem_bytes(EPI);
  constexpr uint32_t BLK = 32 * RB;
  constexpr bool LOADS = EPI == EPI_F32_RESID || EPI == EPI_SWIGLU_BWD;
  constexpr int CPW = EPI == EPI_SWIGLU ? 64 : BN / 2;  // columns per warp
  constexpr int NCH = CPW / 32;                          // 32-column TMEM chunks
  constexpr int UPC = 32 / UNIT;                         // units per chunk
  constexpr int NU = NCH * UPC;
  static_assert((EPI != EPI_SWIGLU && EPI != EPI_CE) || (BN == 256 && STG >= 4096),
                "SwiGLU and CE tiles are 256 wide");
  static_assert(BLK * (EPI == EPI_SWIGLU ? 1 : EPI == EPI_SWIGLU_BWD ? 2 : 1) <= BUF,
                "unit does not fit its staging buffer");
  const Epi& e = p.epi;
  const int lane = st.lane;
  const int row = row0 + lane;
  const bool row_ok = row < p.m_epi;
  const int ncols = EPI == EPI_SWIGLU ? e.half : p.N;
  const int col_w = EPI == EPI_SWIGLU ? nt * 128 + half * 64 : nt * BN + half * (BN / 2);
  const uint32_t tcol_w = EPI == EPI_SWIGLU ? half * 64 : half * (BN / 2);

  auto issue_load = [&](int col, uint32_t bi) {
    if (lane != 0) return;
    const uint32_t b = st.bar + 8 * bi;
    const uint32_t dst = st.a + bi * BUF;
    if constexpr (EPI == EPI_F32_RESID) {
      mbar_arrive_expect_tx(b, BLK);
      tma_load_2d(dst, &om.i1, b, col, row0);
    } else if constexpr (EPI == EPI_SWIGLU_BWD) {
      mbar_arrive_expect_tx(b, 2 * BLK);
      tma_load_2d(dst, &om.i1, b, col, row0);
      tma_load_2d(dst + BLK, &om.i2, b, col, row0);
    }
  };
  if constexpr (LOADS) {
    if (lane == 0) bulk_wait_read0();  // both buffers free
    __syncwarp();
    if (col_w < ncols) issue_load(col_w, ucnt & 1);
  }
  if (!warp_wait(tfull, tfull_ph, p.err)) {
    if constexpr (LOADS) {
      // do not leave the copy into this warp's buffer in flight
      if (col_w < ncols) {
        mbar_wait(st.bar + 8 * (ucnt & 1), (eph >> (ucnt & 1)) & 1u, nullptr);
        eph ^= 1u << (ucnt & 1);
        ++ucnt;
      }
    }
    return false;
  }
  tc_fence_after();

  uint32_t r[32];
  uint32_t r2[EPI == EPI_SWIGLU ? 32 : 1];
  float sq = 0.f;  // F32 / F32_RESID with sq_part: sum of squares of this warp's stored values
  float mx = -INFINITY, sum = 0.f;
  // the target's column within this GEMM (the logits start at vocabulary index col_off)
  const int tgt = ((EPI == EPI_CE || EPI == EPI_CE_GRAD) && row_ok) ? e.targets[row] - e.col_off
                                                                     : -1;
  const float lse_row = (EPI == EPI_CE_GRAD && row_ok) ? e.lse[row] : 0.f;
#pragma unroll 1
  for (int c = 0; c < NCH; ++c) {
    const int ccol = col_w + c * 32;
    if (ccol >= ncols) break;
    tmem_ld32(tbase + tcol_w + c * 32, r);
    if constexpr (EPI == EPI_SWIGLU) tmem_ld32(tbase + 128 + tcol_w + c * 32, r2);
    tmem_ld_wait();
    if constexpr (EPI == EPI_CE) {
      const int nvalid = min(32, p.N - ccol);
      float cm = -INFINITY;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < nvalid) cm = fmaxf(cm, __uint_as_float(r[j]));
      const float nm = fmaxf(mx, cm);
      float acc = sum * __expf(mx - nm);
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < nvalid) acc += __expf(__uint_as_float(r[j]) - nm);
      mx = nm;
      sum = acc;
      if (row_ok && tgt >= ccol && tgt < ccol + nvalid) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j == tgt - ccol) e.tgt_logit[row] = __uint_as_float(r[j]);
      }
      continue;  // statistics only: the logits are not stored
    }
#pragma unroll
    for (int j = 0; j < UPC; ++j) {
      const int u = c * UPC + j;
      const int col = ccol + j * UNIT;
      if (col >= ncols) break;
      const uint32_t bi = ucnt & 1;
      uint8_t* buf = st.p + bi * BUF;
      const uint32_t bufa = st.a + bi * BUF;
      float v[UNIT];
#pragma unroll
      for (int k = 0; k < UNIT; ++k) v[k] = __uint_as_float(r[j * UNIT + k]);
      if constexpr (EPI == EPI_BF16) {
#pragma unroll
        for (int k = 0; k < UNIT; ++k) v[k] *= e.scale;
      }
      if constexpr (EPI == EPI_CE_GRAD) {
        // softmax minus the target's one-hot, from the fp32 logit and the row's LSE
        const int tc = tgt - col;
#pragma unroll
        for (int k = 0; k < UNIT; ++k)
          v[k] = (__expf(v[k] - lse_row) - (k == tc ? 1.f : 0.f)) * e.scale;
      }
      if constexpr (EPI == EPI_F32) {
        // out-of-range rows and columns hold exact zeros (zero-filled operands)
        if (e.sq_part) {
#pragma unroll
          for (int k = 0; k < UNIT; ++k) sq = fmaf(v[k], v[k], sq);
        }
      }
      ++ucnt;
      if constexpr (LOADS) {
        const bool next = u + 1 < NU && col + UNIT < ncols;
        if (next) {
          // the other buffer's last store (the previous unit's) has been read: refill it
          if (lane == 0) bulk_wait_read0();
          __syncwarp();
          issue_load(col + UNIT, bi ^ 1u);
        }
        if (!warp_wait(st.bar + 8 * bi, (eph >> bi) & 1u, p.err)) {
          // do not leave copies into this warp's buffers in flight
          mbar_wait(st.bar + 8 * bi, (eph >> bi) & 1u, nullptr);
          if (next) mbar_wait(st.bar + 8 * (bi ^ 1u), (eph >> (bi ^ 1u)) & 1u, nullptr);
          return false;
        }
        eph ^= 1u << bi;
      } else {
        // this buffer's last store (unit u - 2) has been read
        if (lane == 0) bulk_wait_read1();
        __syncwarp();
      }
      if constexpr (EPI == EPI_F32 || EPI == EPI_F32_RESID || EPI == EPI_BF16 ||
                    EPI == EPI_CE_GRAD) {
        if (col + UNIT > ncols && (ncols & (EPI == EPI_F32 || EPI == EPI_F32_RESID ? 3 : 7))) {
          // a bulk store's bounds check works in 16-byte units, so a last unit
          // whose row end is not 16-byte aligned is written with plain stores
          if constexpr (EPI == EPI_F32_RESID) {
            if (row_ok) {
              const float* res = e.resid + (int64_t)row * e.ld_resid + col;
#pragma unroll
              for (int k = 0; k < UNIT; ++k)
                if (col + k < ncols) {
                  v[k] += res[k];
                  if (e.sq_part) sq = fmaf(v[k], v[k], sq);
                }
            }
          }
          if (row_ok) {
#pragma unroll
            for (int k = 0; k < UNIT; ++k) {
              if (col + k >= ncols) continue;
              if constexpr (EPI == EPI_F32 || EPI == EPI_F32_RESID)
                reinterpret_cast<float*>(e.out)[(int64_t)row * e.ld_out + col + k] = v[k];
              else
                reinterpret_cast<bf16*>(e.out)[(int64_t)row * e.ld_out + col + k] =
                    __float2bfloat16_rn(v[k]);
            }
          }
          continue;
        }
        if constexpr (EPI == EPI_F32_RESID) {
          float q[UNIT];
          get_f32<RB, UNIT>(buf, lane, q);
#pragma unroll
          for (int k = 0; k < UNIT; ++k) v[k] += q[k];
          // out-of-range rows and columns: zero accumulator + zero-filled load
          if (e.sq_part) {
#pragma unroll
            for (int k = 0; k < UNIT; ++k) sq = fmaf(v[k], v[k], sq);
          }
        }
        if constexpr (EPI == EPI_F32 || EPI == EPI_F32_RESID) put_f32<RB, UNIT>(buf, lane, v);
        else put_bf16<RB, UNIT>(buf, lane, v);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&om.o1, bufa, col, row0);
          bulk_commit();
        }
      } else if constexpr (EPI == EPI_SWIGLU) {
        // three 2 KB outputs per 32-column unit: g and u fill the warp's whole
        // 4 KB staging, then s (fewer, larger bulk stores than double buffering
        // narrower units)
        float uu[UNIT], sv[UNIT];
#pragma unroll
        for (int k = 0; k < UNIT; ++k) {
          uu[k] = __uint_as_float(r2[j * UNIT + k]);
          sv[k] = silu_f(v[k]) * uu[k];
        }
        if (lane == 0) bulk_wait_read0();
        __syncwarp();
        put_bf16<RB, UNIT>(st.p, lane, v);
        put_bf16<RB, UNIT>(st.p + BLK, lane, uu);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&om.o1, st.a, col, row0);
          tma_store_2d(&om.o2, st.a + BLK, col, row0);
          bulk_commit();
          bulk_wait_read0();
        }
        __syncwarp();
        put_bf16<RB, UNIT>(st.p, lane, sv);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&om.o3, st.a, col, row0);
          bulk_commit();
        }
      } else if constexpr (EPI == EPI_SWIGLU_BWD) {
        // ds (accumulator) with the saved g, u -> dg = ds u silu'(g), du = ds silu(g)
        float g[UNIT], uu[UNIT], dg[UNIT], du[UNIT];
        get_bf16<RB, UNIT>(buf, lane, g);
        get_bf16<RB, UNIT>(buf + BLK, lane, uu);
#pragma unroll
        for (int k = 0; k < UNIT; ++k) {
          const float sg = 1.0f / (1.0f + __expf(-g[k]));
          dg[k] = v[k] * uu[k] * sg * (1.0f + g[k] * (1.0f - sg));
          du[k] = v[k] * g[k] * sg;
        }
        put_bf16<RB, UNIT>(buf, lane, dg);
        put_bf16<RB, UNIT>(buf + BLK, lane, du);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&om.o1, bufa, col, row0);
          tma_store_2d(&om.o2, bufa + BLK, col, row0);
          bulk_commit();
        }
      }
    }
  }
  if constexpr (EPI == EPI_CE) {
    if (row_ok) e.part[(int64_t)row * e.part_ld + 2 * nt + half] = make_float2(mx, sum);
  }
  if constexpr (EPI == EPI_F32 || EPI == EPI_F32_RESID) {
    if (e.sq_part) {
      double d = sq;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
      if (lane == 0) e.sq_part[(int64_t)tile * p.sq_slots + slot] = d;
    }
  }
  return true;
}

// ----------------------------------------------------------------- kernel
template <int A_MN, int B_MN, int EPI, int BN>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tma_a,
                const __grid_constant__ CUtensorMap tma_b, const __grid_constant__ OutMaps om,
                const GemmParams p) {
  constexpr int STAGES = Tile<BN>::STAGES;
  constexpr uint32_t STAGE_BYTES = Tile<BN>::STAGE_BYTES;
  using OS = OutStage<BN, false>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Tile<BN>::OFF_OUT + OS::TOTAL);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain, epilogue inputs[8][2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 21);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * STAGES;
  const uint32_t tfull0 = empty0 + 8 * STAGES;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain = tempty0 + 16;
  const uint32_t ebar0 = drain + 8;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, EPI_THREADS / 32);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    for (int i = 0; i < 16; ++i) mbar_init(ebar0 + 8 * i, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tma_a);
    tma_prefetch_desc(&tma_b);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int ntiles = p.m_tiles * p.n_tiles;
  const int nunits = ntiles * p.splits;
  const uint32_t smem_base = smem_u32(smem);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t ph = 0;
      uint32_t pending = 0, pending_par = 0;  // stages with a load in flight
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        int mt, nt;
        tile_coords(u % ntiles, p, mt, nt);
        const int m0 = mt * BM;
        const int kb0 = (u / ntiles) * p.kb_split;
        const int kb1 = min(p.k_blocks, kb0 + p.kb_split);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, ph ^ 1, p.err)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + 8 * stage;
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          const uint32_t sa = smem_base + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          const int k0 = kb * BK;
          if (A_MN) {
            tma_load_2d(sa, &tma_a, fb, m0, k0);
            tma_load_2d(sa + MN_CHUNK_BYTES, &tma_a, fb, m0 + 64, k0);
          } else {
            tma_load_2d(sa, &tma_a, fb, k0, m0);
          }
          if (B_MN) {
            const int n0 = nt * BN;
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_2d(sb + j * MN_CHUNK_BYTES, &tma_b, fb, n0 + 64 * j, k0);
          } else {
            // 64-row boxes; SwiGLU stacks gate rows nt*128+[0,128) and up rows
            // half+nt*128+[0,128) into one 256-row tile
#pragma unroll
            for (int j = 0; j < BN / 64; ++j) {
              const int r = (EPI == EPI_SWIGLU) ? nt * 128 + (j & 1) * 64 + (j >> 1) * p.swiglu_half
                                                : nt * BN + j * 64;
              tma_load_2d(sb + j * MN_CHUNK_BYTES, &tma_b, fb, k0, r);
            }
          }
          pending |= 1u << stage;
          pending_par = (pending_par & ~(1u << stage)) | (ph << stage);
          if (++stage == STAGES) {
            stage = 0;
            ph ^= 1;
          }
        }
      }
      if (!ok) {
        // do not leave while copies into this CTA's shared memory are in flight
        for (int s = 0; s < STAGES; ++s)
          if (pending & (1u << s)) mbar_wait(full0 + 8 * s, (pending_par >> s) & 1u, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------------- MMA
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, A_MN, B_MN);
      const uint64_t a_desc0 = sdesc_sw128(smem_base, A_MN ? MN_CHUNK_BYTES : 16, 1024);
      const uint64_t b_desc0 = sdesc_sw128(smem_base + A_BYTES, B_MN ? MN_CHUNK_BYTES : 16, 1024);
      int stage = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t acc_ph = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        if (!mbar_wait(tempty0 + 8 * acc, acc_ph ^ 1, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        const int kb0 = (u / ntiles) * p.kb_split;
        const int kb1 = min(p.k_blocks, kb0 + p.kb_split);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, ph, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // descriptors of this stage: the ring's first stage plus the stage
          // offset, then one K=16 step = 32 B (K-major) or 2048 B (MN-major)
          const uint64_t ad0 = a_desc0 + static_cast<uint64_t>(stage) * (STAGE_BYTES >> 4);
          const uint64_t bd0 = b_desc0 + static_cast<uint64_t>(stage) * (STAGE_BYTES >> 4);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = ad0 + static_cast<uint64_t>(k) * ((A_MN ? 2048 : 32) >> 4);
            const uint64_t bd = bd0 + static_cast<uint64_t>(k) * ((B_MN ? 2048 : 32) >> 4);
            tc_mma_bf16(d_tmem, ad, bd, idesc, kb != kb0 || k != 0);
          }
          tc_commit(empty0 + 8 * stage);
          if (++stage == STAGES) {
            stage = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(tfull0 + 8 * acc);
        acc ^= 1;
        if (acc == 0) acc_ph ^= 1;
      }
      // make sure no MMA is still writing TMEM before it is released
      tc_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;             // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;   // which half of the tile's columns
    uint8_t* stg = smem + Tile<BN>::OFF_OUT + (warp - 2) * OS::BYTES;
    const Stage st{stg, smem_u32(stg), ebar0 + 16 * (warp - 2), lane};
    uint32_t ucnt = 0, eph = 0;
    int acc = 0;
    uint32_t acc_ph = 0;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
      int mt, nt;
      const int t = u % ntiles;
      tile_coords(t, p, mt, nt);
      const int row0 = (u / ntiles) * p.m_pad + mt * BM + q * 32;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      if (!epilogue_tile<EPI, BN, OS::BYTES>(p, om, tbase, row0, nt, half, st, ucnt, eph,
                                             tfull0 + 8 * acc, acc_ph, t, warp - 2))
        break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
      acc ^= 1;
      if (acc == 0) acc_ph ^= 1;
    }
    if (lane == 0) bulk_wait0();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------- NF4 kernel
// The single-CTA GEMM with a frozen NF4 weight as its B operand, decoded into
// the shared-memory tile on the way (no bf16 copy of the weight exists), plus
// an optional tail k-block of ordinary bf16 operands (the LoRA term folded in
// as extra K: [X | U] [W | B]^T forward, [dY | dU] [W ; A] backward).
//
// W is [rows, cols] row-major with two 4-bit codes per byte (element 2j in the
// low nibble of byte j) and one fp32 scale per 64 consecutive elements of a
// row (cols % 256 == 0, so each 64-element block lies in one row and the
// scale array's row stride is a multiple of 16 bytes). K-major use (forward,
// B(n, k) = W[n][k]) and MN-major use (dX, B(n, k) = W[k][n]) both decode one
// 64-element block into one 128-byte row of the 128-byte-swizzled tile.
//
// Roles (448 threads): warp 0 TMA producer (A, the codes [64 rows x 32 B or
// 64 rows x 128 B boxes] and the scales [64 rows x 4 fp32] of each stage into
// a raw area of the stage; the tail's A and B straight into the tile), warp 1
// MMA, warps 2-9 epilogue (as above), warps 10-13 decode: wait for a stage's
// raw bytes, turn them into the bf16 B tile, and arrive on the stage's full
// barrier, which the MMA waits for.
constexpr int NF4_THREADS = 448;
// The pair kernel runs two decode groups of 4 warps (warps 10-13 and 14-17)
// that take alternate k-blocks, so one group's decode latency (the permute
// chains, the proxy fence, the arrive) overlaps the other's.
constexpr int NF4P_THREADS = 576;
constexpr int NF4_BN = 256;

struct TileN4 {
  static constexpr uint32_t B_BYTES = NF4_BN * BK * 2;                  // 32 KB
  static constexpr uint32_t CODE_BYTES = NF4_BN * BK / 2;               // 8 KB
  static constexpr uint32_t ABS_BYTES = 4096;                           // <= 256 rows x 16 B
  static constexpr uint32_t OFF_B = A_BYTES;
  static constexpr uint32_t OFF_CODE = OFF_B + B_BYTES;
  static constexpr uint32_t OFF_ABS = OFF_CODE + CODE_BYTES;
  static constexpr uint32_t STAGE_BYTES = OFF_ABS + ABS_BYTES;          // 60 KB
  static constexpr int STAGES = 3;
  static constexpr uint32_t OFF_OUT = STAGES * STAGE_BYTES;
  static constexpr size_t SMEM = OFF_OUT + OutStage<NF4_BN, false>::TOTAL + 1024 + 512;
};

// Codes / scales maps of the NF4 operand and the tail's A.
struct Nf4Maps {
  CUtensorMap codes, scales, a2;
};

// The sixteen NormalFloat-4 levels (QLoRA), ascending by code.
__constant__ float kNf4Levels[16] = {
    -1.0f, -0.6961928009986877f, -0.5250730514526367f, -0.39491748809814453f,
    -0.28444138169288635f, -0.18477343022823334f, -0.09105003625154495f, 0.0f,
    0.07958029955625534f, 0.16093020141124725f, 0.24611230194568634f, 0.33791524171829224f,
    0.44070982933044434f, 0.5626170039176941f, 0.7229568362236023f, 1.0f};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// The 16 products T[c] = bf16(level[c] * sc) of one 64-weight block, as byte
// planes: lo[q] holds the low bytes of T[4q .. 4q+3], hi[q] the high bytes.
__device__ __forceinline__ void nf4_planes(float sc, uint32_t (&lo)[4], uint32_t (&hi)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t p0 = pack_bf16x2(kNf4Levels[4 * q] * sc, kNf4Levels[4 * q + 1] * sc);
    const uint32_t p1 = pack_bf16x2(kNf4Levels[4 * q + 2] * sc, kNf4Levels[4 * q + 3] * sc);
    lo[q] = prmt(p0, p1, 0x6420);
    hi[q] = prmt(p0, p1, 0x7531);
  }
}

// Multipliers that stand in for shifts (w * 16 = w << 4; umulhi(w, 2^16) =
// w >> 16; umulhi(w, 2^20) = w >> 12): kept in constant memory so the
// compiler issues integer multiplies, which run on the FMA pipe, and the
// byte permutes and logic ops have the ALU pipe to themselves.
__constant__ uint32_t kNf4ShiftMul[3] = {16u, 1u << 16, 1u << 20};

// T[c] for the four codes in the low 16 bits of s (code j in bits 4j..4j+3)
// as two bf16 pairs (code 0 in the low half of .x). sx = s with bit 3 of
// every code flipped; t = s << 4 (the bytes of s and t carry the top bits
// of the four codes). A byte permute indexes 8 bytes, so each plane is looked
// up in its lower (codes 0-7, selector s) and upper (8-15, selector sx)
// halves and the two merged on bit 3 of the code, replicated into a byte
// mask by the permute's sign mode.
__device__ __forceinline__ uint2 nf4_lookup4(uint32_t s, uint32_t sx, uint32_t t,
                                             const uint32_t (&lo)[4], const uint32_t (&hi)[4]) {
  const uint32_t m = prmt(t, s, 0xD9C8);
  const uint32_t la = prmt(lo[0], lo[1], s), lb = prmt(lo[2], lo[3], sx);
  const uint32_t ha = prmt(hi[0], hi[1], s), hb = prmt(hi[2], hi[3], sx);
  const uint32_t l = (la & ~m) | (lb & m);
  const uint32_t h = (ha & ~m) | (hb & m);
  return make_uint2(prmt(l, h, 0x5140), prmt(l, h, 0x7362));
}

// The eight weights of one code word (element j in bits 4j..4j+3) as bf16.
__device__ __forceinline__ uint4 nf4_lookup8(uint32_t w, const uint32_t (&lo)[4],
                                             const uint32_t (&hi)[4]) {
  const uint32_t sxw = w ^ 0x88888888u;
  const uint2 e0 = nf4_lookup4(w, sxw, w * kNf4ShiftMul[0], lo, hi);
  const uint2 e1 = nf4_lookup4(__umulhi(w, kNf4ShiftMul[1]), __umulhi(sxw, kNf4ShiftMul[1]),
                               __umulhi(w, kNf4ShiftMul[2]), lo, hi);
  return make_uint4(e0.x, e0.y, e1.x, e1.y);
}

// Decode one 64-weight run (32 code bytes as two 16-byte chunks c0, c1; one
// scale) into the 128-byte row `row` of a 128-byte-swizzled bf16 tile at dst.
__device__ __forceinline__ void nf4_decode_run(uint4 c0, uint4 c1, float sc, uint8_t* dst,
                                               int row) {
  uint32_t lo[4], hi[4];
  nf4_planes(sc, lo, hi);
  const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
  for (int c8 = 0; c8 < 8; ++c8) {
    // 4 code bytes = 8 weights, element 2j in the low nibble of byte j
    *reinterpret_cast<uint4*>(dst + sw128_offset(row, c8)) = nf4_lookup8(w[c8], lo, hi);
  }
}

template <int B_MN, int EPI>
__global__ void __launch_bounds__(NF4_THREADS, 1)
    gemm_nf4_kernel(const __grid_constant__ CUtensorMap tma_a,
                    const __grid_constant__ CUtensorMap tma_b2,
                    const __grid_constant__ Nf4Maps nm, const __grid_constant__ OutMaps om,
                    const GemmParams p) {
  constexpr int BN = NF4_BN;
  constexpr int STAGES = TileN4::STAGES;
  constexpr uint32_t STAGE_BYTES = TileN4::STAGE_BYTES;
  using OS = OutStage<BN, false>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + TileN4::OFF_OUT + OS::TOTAL);
  // bars: raw[S], full[S], empty[S], tfull[2], tempty[2], drain, epilogue inputs[8][2];
  // then the TMEM address
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 21);
  const uint32_t raw0 = smem_u32(bars);
  const uint32_t full0 = raw0 + 8 * STAGES;
  const uint32_t empty0 = full0 + 8 * STAGES;
  const uint32_t tfull0 = empty0 + 8 * STAGES;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain = tempty0 + 16;
  const uint32_t ebar0 = drain + 8;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(raw0 + 8 * s, 1);
      mbar_init(full0 + 8 * s, 4);  // one arrival per decode warp
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, EPI_THREADS / 32);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < 16; ++i) mbar_init(ebar0 + 8 * i, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tma_a);
    tma_prefetch_desc(&tma_b2);
    tma_prefetch_desc(&nm.codes);
    tma_prefetch_desc(&nm.scales);
    tma_prefetch_desc(&nm.a2);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int ntiles = p.m_tiles * p.n_tiles;
  const uint32_t smem_base = smem_u32(smem);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t ph = 0;
      uint32_t pending = 0, pending_par = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        int mt, nt;
        tile_coords(t, p, mt, nt);
        const int m0 = mt * BM;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, ph ^ 1, p.err)) {
            ok = false;
            break;
          }
          const uint32_t rb = raw0 + 8 * stage;
          const uint32_t sa = smem_base + stage * STAGE_BYTES;
          const uint32_t sb = sa + TileN4::OFF_B;
          const uint32_t sc = sa + TileN4::OFF_CODE;
          const uint32_t ss = sa + TileN4::OFF_ABS;
          const int k0 = kb * BK;
          if (kb < p.kb_main) {
            mbar_arrive_expect_tx(rb, A_BYTES + (B_MN ? 64 * 128 + 64 * 16
                                                       : TileN4::CODE_BYTES + NF4_BN * 16));
            tma_load_2d(sa, &tma_a, rb, k0, m0);
            if (B_MN) {
              // W rows k0..k0+63, columns nt*256..: 128 code bytes and 4 scales per row
              tma_load_2d(sc, &nm.codes, rb, nt * (BN / 2), k0);
              tma_load_2d(ss, &nm.scales, rb, nt * (BN / 64), k0);
            } else {
#pragma unroll
              for (int j = 0; j < BN / 64; ++j) {
                const int r = (EPI == EPI_SWIGLU)
                                  ? nt * 128 + (j & 1) * 64 + (j >> 1) * p.swiglu_half
                                  : nt * BN + j * 64;
                tma_load_2d(sc + j * 2048, &nm.codes, rb, k0 / 2, r);
                tma_load_2d(ss + j * 1024, &nm.scales, rb, kb & ~3, r);
              }
            }
          } else {
            // tail: ordinary bf16 A and B for k beyond the decoded operand
            const int kt = k0 - p.kb_main * BK;
            mbar_arrive_expect_tx(rb, A_BYTES + TileN4::B_BYTES);
            tma_load_2d(sa, &nm.a2, rb, kt, m0);
#pragma unroll
            for (int j = 0; j < BN / 64; ++j) {
              if (B_MN) {
                tma_load_2d(sb + j * MN_CHUNK_BYTES, &tma_b2, rb, nt * BN + 64 * j, kt);
              } else {
                const int r = (EPI == EPI_SWIGLU)
                                  ? nt * 128 + (j & 1) * 64 + (j >> 1) * p.swiglu_half
                                  : nt * BN + j * 64;
                tma_load_2d(sb + j * MN_CHUNK_BYTES, &tma_b2, rb, kt, r);
              }
            }
          }
          pending |= 1u << stage;
          pending_par = (pending_par & ~(1u << stage)) | (ph << stage);
          if (++stage == STAGES) {
            stage = 0;
            ph ^= 1;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < STAGES; ++s)
          if (pending & (1u << s)) mbar_wait(raw0 + 8 * s, (pending_par >> s) & 1u, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------------- MMA
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, 0, B_MN);
      const uint64_t a_desc0 = sdesc_sw128(smem_base, 16, 1024);
      const uint64_t b_desc0 =
          sdesc_sw128(smem_base + TileN4::OFF_B, B_MN ? MN_CHUNK_BYTES : 16, 1024);
      int stage = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t acc_ph = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        if (!mbar_wait(tempty0 + 8 * acc, acc_ph ^ 1, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, ph, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad0 = a_desc0 + static_cast<uint64_t>(stage) * (STAGE_BYTES >> 4);
          const uint64_t bd0 = b_desc0 + static_cast<uint64_t>(stage) * (STAGE_BYTES >> 4);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = ad0 + static_cast<uint64_t>(k) * (32 >> 4);
            const uint64_t bd = bd0 + static_cast<uint64_t>(k) * ((B_MN ? 2048 : 32) >> 4);
            tc_mma_bf16(d_tmem, ad, bd, idesc, (kb | k) != 0);
          }
          tc_commit(empty0 + 8 * stage);
          if (++stage == STAGES) {
            stage = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(tfull0 + 8 * acc);
        acc ^= 1;
        if (acc == 0) acc_ph ^= 1;
      }
      tc_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    uint8_t* stg = smem + TileN4::OFF_OUT + (warp - 2) * OS::BYTES;
    const Stage st{stg, smem_u32(stg), ebar0 + 16 * (warp - 2), lane};
    uint32_t ucnt = 0, eph = 0;
    int acc = 0;
    uint32_t acc_ph = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      int mt, nt;
      tile_coords(t, p, mt, nt);
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      if (!epilogue_tile<EPI, BN, OS::BYTES>(p, om, tbase, mt * BM + q * 32, nt, half, st, ucnt,
                                             eph, tfull0 + 8 * acc, acc_ph, t, warp - 2))
        break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
      acc ^= 1;
      if (acc == 0) acc_ph ^= 1;
    }
    if (lane == 0) bulk_wait0();
    __syncwarp();
  } else {
    // -------------------------------------------------------------- decode
    const int dt = static_cast<int>(threadIdx.x) - 320;  // 0..127
    int stage = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      for (int kb = 0; kb < p.k_blocks; ++kb) {
        if (!warp_wait(raw0 + 8 * stage, ph, p.err)) {
          ok = false;
          break;
        }
        if (kb < p.kb_main) {
          uint8_t* sp = smem + stage * STAGE_BYTES;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int u = dt + 128 * i;  // one 64-element block of W per u
            if (B_MN) {
              // W row k0 + k_row, columns ch*64..: 32 code bytes in a 128-byte-swizzled row
              const int k_row = u & 63, ch = u >> 6;
              const uint8_t* cr = sp + TileN4::OFF_CODE + k_row * 128;
              const uint4 c0 = *reinterpret_cast<const uint4*>(cr + (((2 * ch) ^ (k_row & 7)) << 4));
              const uint4 c1 =
                  *reinterpret_cast<const uint4*>(cr + (((2 * ch + 1) ^ (k_row & 7)) << 4));
              const float sc =
                  *reinterpret_cast<const float*>(sp + TileN4::OFF_ABS + k_row * 16 + ch * 4);
              nf4_decode_run(c0, c1, sc, sp + TileN4::OFF_B + ch * MN_CHUNK_BYTES, k_row);
            } else {
              const uint4* cr = reinterpret_cast<const uint4*>(sp + TileN4::OFF_CODE + u * 32);
              const float sc = *reinterpret_cast<const float*>(sp + TileN4::OFF_ABS + u * 16 +
                                                               (kb & 3) * 4);
              nf4_decode_run(cr[0], cr[1], sc, sp + TileN4::OFF_B, u);
            }
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(full0 + 8 * stage);
        if (++stage == STAGES) {
          stage = 0;
          ph ^= 1;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------- NF4 pair kernel
// The NF4 GEMM on CTA pairs (clusters of 2, tcgen05.mma.cta_group::2 with
// 256 x 256 x 16 tiles): each CTA stages its own 128 rows of A and decodes
// only its 128 of the tile's 256 B columns, half the decode work per MMA
// flop of the single-CTA kernel. TMA brings each CTA's codes and scales to a
// local "raw" barrier; A (and the tail's A2 / B2) complete on the even CTA's
// "full" barrier, on which both CTAs' decode warps also arrive after a
// generic-to-async proxy fence over their decoded tiles. The even CTA's MMA
// thread commits to both CTAs' "empty" barriers; the epilogue is the pair
// GEMM's.
struct TileN4P {
  static constexpr int BH = NF4_BN / 2;                      // B columns per CTA
  static constexpr uint32_t B_BYTES = BH * BK * 2;           // 16 KB
  static constexpr uint32_t CODE_BYTES = BH * BK / 2;        // 4 KB
  static constexpr uint32_t ABS_BYTES = 2048;                // <= 128 rows x 16 B
  static constexpr uint32_t OFF_B = A_BYTES;
  static constexpr uint32_t OFF_CODE = OFF_B + B_BYTES;
  static constexpr uint32_t OFF_ABS = OFF_CODE + CODE_BYTES;
  static constexpr uint32_t STAGE_BYTES = OFF_ABS + ABS_BYTES;  // 38 KB
  static constexpr int STAGES = 5;
  static constexpr uint32_t OFF_OUT = STAGES * STAGE_BYTES;
  static constexpr size_t SMEM = OFF_OUT + OutStage<NF4_BN, true>::TOTAL + 1024 + 512;
};
static_assert(TileN4P::SMEM <= 232448, "NF4 pair tile exceeds the shared memory of a CTA");
static_assert(TileN4P::STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte swizzle alignment");

template <int B_MN, int EPI>
__global__ void __launch_bounds__(NF4P_THREADS, 1)
    gemm2_nf4_kernel(const __grid_constant__ CUtensorMap tma_a,
                     const __grid_constant__ CUtensorMap tma_b2,
                     const __grid_constant__ Nf4Maps nm, const __grid_constant__ OutMaps om,
                     const GemmParams p) {
  constexpr int BN = NF4_BN;
  constexpr int BH = TileN4P::BH;
  constexpr int STAGES = TileN4P::STAGES;
  constexpr uint32_t STAGE_BYTES = TileN4P::STAGE_BYTES;
  using OS = OutStage<BN, true>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + TileN4P::OFF_OUT + OS::TOTAL);
  // bars: raw[2][S] (one set per decode group), full[S], empty[S], tfull[2],
  // tempty[2], drain, epilogue inputs[8][2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 4 * STAGES + 21);
  const uint32_t raw0 = smem_u32(bars);
  const uint32_t full0 = raw0 + 8 * 2 * STAGES;
  const uint32_t empty0 = full0 + 8 * STAGES;
  const uint32_t tfull0 = empty0 + 8 * STAGES;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain = tempty0 + 16;
  const uint32_t ebar0 = drain + 8;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the pair MMAs
  const int pair = static_cast<int>(blockIdx.x) >> 1;
  const int npairs = static_cast<int>(gridDim.x) >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2 * STAGES; ++s) mbar_init(raw0 + 8 * s, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1 + 2 * 4);  // even producer + both CTAs' decode warps
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 2 * (EPI_THREADS / 32));
    }
    mbar_init(drain, 1);
    for (int i = 0; i < 16; ++i) mbar_init(ebar0 + 8 * i, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tma_a);
    tma_prefetch_desc(&tma_b2);
    tma_prefetch_desc(&nm.codes);
    tma_prefetch_desc(&nm.scales);
    tma_prefetch_desc(&nm.a2);
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t full_even = mapa_shared(full0, 0);
  const uint32_t tempty_even = mapa_shared(tempty0, 0);

  const int ntiles = p.m_tiles * p.n_tiles;  // m_tiles counts 256-row pair tiles
  const int nunits = ntiles * p.splits;       // tiles x K-slices
  const uint32_t smem_base = smem_u32(smem);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t ph = 0;
      uint32_t it = 0;  // k-blocks issued, across units: group it & 1 decodes it
      bool ok = true;
      for (int u = pair; u < nunits && ok; u += npairs) {
        int mt, nt;
        tile_coords(u % ntiles, p, mt, nt);
        const int m0 = (2 * mt + static_cast<int>(rank)) * BM;
        const int kb0 = (u / ntiles) * p.kb_split;
        const int kb1 = min(p.k_blocks, kb0 + p.kb_split);
        // first of this CTA's 128 B rows (K-major) / columns (MN-major)
        const int r0 = (EPI == EPI_SWIGLU) ? nt * 128 + static_cast<int>(rank) * p.swiglu_half
                                           : nt * BN + static_cast<int>(rank) * BH;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          if (!mbar_wait(empty0 + 8 * stage, ph ^ 1, p.err)) {
            ok = false;
            break;
          }
          const uint32_t rb = raw0 + 8 * ((it & 1) * STAGES + stage);
          const uint32_t fb = full_even + 8 * stage;
          const uint32_t sa = smem_base + stage * STAGE_BYTES;
          const uint32_t sb = sa + TileN4P::OFF_B;
          const uint32_t sc = sa + TileN4P::OFF_CODE;
          const uint32_t ss = sa + TileN4P::OFF_ABS;
          const int k0 = kb * BK;
          if (kb < p.kb_main) {
            if (rank == 0) mbar_arrive_expect_tx(full0 + 8 * stage, 2 * A_BYTES);
            tma_load_2d_pair(sa, &tma_a, fb, k0, m0);
            if (B_MN) {
              // W rows k0..k0+63, this CTA's 128 columns: 64 code bytes and the
              // 4 scales of the tile's 256 columns per row
              mbar_arrive_expect_tx(rb, 64 * 64 + 64 * 16);
              tma_load_2d(sc, &nm.codes, rb, r0 / 2, k0);
              tma_load_2d(ss, &nm.scales, rb, nt * (BN / 64), k0);
            } else {
              // this CTA's 128 W rows, 32 code bytes and 4 scales each, 64 rows per box
              mbar_arrive_expect_tx(rb, TileN4P::CODE_BYTES + BH * 16);
#pragma unroll
              for (int j = 0; j < BH / 64; ++j) {
                tma_load_2d(sc + j * 2048, &nm.codes, rb, k0 / 2, r0 + 64 * j);
                tma_load_2d(ss + j * 1024, &nm.scales, rb, kb & ~3, r0 + 64 * j);
              }
            }
          } else {
            // tail: ordinary bf16 A2 and B2; the decode warps only pass through
            const int kt = k0 - p.kb_main * BK;
            if (rank == 0) mbar_arrive_expect_tx(full0 + 8 * stage, 2 * (A_BYTES + TileN4P::B_BYTES));
            tma_load_2d_pair(sa, &nm.a2, fb, kt, m0);
#pragma unroll
            for (int j = 0; j < BH / 64; ++j) {
              if (B_MN)
                tma_load_2d_pair(sb + j * MN_CHUNK_BYTES, &tma_b2, fb, r0 + 64 * j, kt);
              else
                tma_load_2d_pair(sb + j * MN_CHUNK_BYTES, &tma_b2, fb, kt, r0 + 64 * j);
            }
            mbar_arrive(rb);
          }
          if (++stage == STAGES) {
            stage = 0;
            ph ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ----------------------------------------------------------------- MMA
      constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN, 0, B_MN);
      const uint64_t a_desc0 = sdesc_sw128(smem_base, 16, 1024);
      const uint64_t b_desc0 =
          sdesc_sw128(smem_base + TileN4P::OFF_B, B_MN ? MN_CHUNK_BYTES : 16, 1024);
      int stage = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t acc_ph = 0;
      bool ok = true;
      for (int u = pair; u < nunits && ok; u += npairs) {
        if (!mbar_wait_cluster(tempty0 + 8 * acc, acc_ph ^ 1, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        const int kb0 = (u / ntiles) * p.kb_split;
        const int kb1 = min(p.k_blocks, kb0 + p.kb_split);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, ph, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad0 = a_desc0 + static_cast<uint64_t>(stage) * (STAGE_BYTES >> 4);
          const uint64_t bd0 = b_desc0 + static_cast<uint64_t>(stage) * (STAGE_BYTES >> 4);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = ad0 + static_cast<uint64_t>(k) * (32 >> 4);
            const uint64_t bd = bd0 + static_cast<uint64_t>(k) * ((B_MN ? 2048 : 32) >> 4);
            tc_mma_bf16_pair(d_tmem, ad, bd, idesc, kb != kb0 || k != 0);
          }
          tc_commit_pair_mc(empty0 + 8 * stage, 0x3);
          if (++stage == STAGES) {
            stage = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(tfull0 + 8 * acc, 0x3);
        acc ^= 1;
        if (acc == 0) acc_ph ^= 1;
      }
      tc_commit_pair(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    uint8_t* stg = smem + TileN4P::OFF_OUT + (warp - 2) * OS::BYTES;
    const Stage st{stg, smem_u32(stg), ebar0 + 16 * (warp - 2), lane};
    uint32_t ucnt = 0, eph = 0;
    int acc = 0;
    uint32_t acc_ph = 0;
    for (int u = pair; u < nunits; u += npairs) {
      int mt, nt;
      const int t = u % ntiles;
      tile_coords(t, p, mt, nt);
      const int mrow = 2 * mt + static_cast<int>(rank);
      const int row0 = (u / ntiles) * p.m_pad + mrow * BM + q * 32;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      if (!epilogue_tile<EPI, BN, OS::BYTES>(p, om, tbase, row0, nt, half, st,
                                             ucnt, eph, tfull0 + 8 * acc, acc_ph, t,
                                             static_cast<int>(rank) * 8 + (warp - 2)))
        break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_even + 8 * acc);
      acc ^= 1;
      if (acc == 0) acc_ph ^= 1;
    }
    if (lane == 0) bulk_wait0();
    __syncwarp();
  } else {
    // -------------------------------------------------------------- decode
    const int dg = static_cast<int>(threadIdx.x) - 320;
    const int dt = dg & 127;  // thread within the group
    const uint32_t grp = static_cast<uint32_t>(dg >> 7);
    int stage = 0;
    uint32_t it = 0;  // k-blocks this CTA has passed, across units
    bool ok = true;
    for (int u = pair; u < nunits && ok; u += npairs) {
      const int kb0 = (u / ntiles) * p.kb_split;
      const int kb1 = min(p.k_blocks, kb0 + p.kb_split);
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        if ((it & 1) != grp) {  // the other group's k-block
          if (++stage == STAGES) stage = 0;
          continue;
        }
        // this group's raw barrier of the stage: the group's uses of it are the
        // k-blocks it = c + 2 S n (one residue c mod 2 S), use n completing its
        // phase n, so the group sees every phase in order (with one barrier
        // per stage and S odd, a group would skip phases, and a parity wait
        // could pass on the phase before the one it waits for)
        if (!warp_wait(raw0 + 8 * (grp * STAGES + stage), (it / (2 * STAGES)) & 1, p.err)) {
          ok = false;
          break;
        }
        if (kb < p.kb_main) {
          uint8_t* sp = smem + stage * STAGE_BYTES;
          if (B_MN) {
            // W row k0 + k_row, this CTA's columns ch*64..: 32 of the row's 64
            // code bytes, 64-byte-swizzled
            const int k_row = dt & 63, ch = dt >> 6;
            const uint8_t* cr = sp + TileN4P::OFF_CODE + k_row * 64;
            const int sw = (k_row >> 1) & 3;
            const uint4 c0 = *reinterpret_cast<const uint4*>(cr + (((2 * ch) ^ sw) << 4));
            const uint4 c1 = *reinterpret_cast<const uint4*>(cr + (((2 * ch + 1) ^ sw) << 4));
            const float sc = *reinterpret_cast<const float*>(
                sp + TileN4P::OFF_ABS + k_row * 16 + (static_cast<int>(rank) * 2 + ch) * 4);
            nf4_decode_run(c0, c1, sc, sp + TileN4P::OFF_B + ch * MN_CHUNK_BYTES, k_row);
          } else {
            const uint4* cr = reinterpret_cast<const uint4*>(sp + TileN4P::OFF_CODE + dt * 32);
            const float sc = *reinterpret_cast<const float*>(sp + TileN4P::OFF_ABS + dt * 16 +
                                                             (kb & 3) * 4);
            nf4_decode_run(cr[0], cr[1], sc, sp + TileN4P::OFF_B, dt);
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(full_even + 8 * stage);
        if (++stage == STAGES) stage = 0;
      }
    }
  }

  tc_fence_before();
  cluster_sync();
  if (p.err && *reinterpret_cast<volatile int*>(p.err) != 0) {
    // after a timed-out wait, copies issued just before may still be landing
    // on this pair's shared memory: let them finish before the CTAs exit
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 200000ull) {
    }
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------ pair kernel
// The same GEMM on CTA pairs (clusters of 2) with the pair MMA
// (tcgen05.mma.cta_group::2, 256 x 256 x 16): each CTA loads its own 128 rows
// of A and 128 of the tile's 256 columns of B, i.e. 32 KB per 64-deep stage
// instead of the 48 KB a single-CTA 128 x 256 tile needs for the same flops -
// one third less shared-memory fill per flop, and 6 stages of lookahead.
// The even CTA's producer arms its full barrier for both CTAs' bytes and both
// producers' TMA copies complete on it; its lane-0 MMA thread issues the pair
// MMAs and commits (multicast) to both CTAs' empty / accumulator-full
// barriers; every epilogue warp of both CTAs hands its accumulator back on the
// even CTA's accumulator-empty barrier. Each CTA's epilogue reads the 128 rows
// of the tile its own TMEM holds, with the same epilogues as above.
template <int BN_>
struct Tile2 {
  static_assert(BN_ == 256, "pair tiles are 256 x 256 (256 x 192 pairs measured slower than 128 x 192 single tiles)");
  static constexpr int BN = BN_;      // pair tile width (N of the MMA)
  static constexpr int BH = BN / 2;   // columns of B each CTA loads
  static constexpr uint32_t B_BYTES = BH * BK * 2;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;  // 32 KB
  static constexpr int STAGES = 6;
  static constexpr uint32_t OFF_OUT = STAGES * STAGE_BYTES;
  static constexpr size_t SMEM = OFF_OUT + OutStage<BN, true>::TOTAL + 1024 + 512;
};

template <int A_MN, int B_MN, int EPI, int BN>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm2_kernel(const __grid_constant__ CUtensorMap tma_a,
                 const __grid_constant__ CUtensorMap tma_b, const __grid_constant__ OutMaps om,
                 const GemmParams p) {
  using TL = Tile2<BN>;
  constexpr int STAGES = TL::STAGES;
  constexpr int BH = TL::BH;
  constexpr uint32_t STAGE_BYTES = TL::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  using OS = OutStage<BN, true>;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + TL::OFF_OUT + OS::TOTAL);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain, epilogue inputs[8][2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 21);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * STAGES;
  const uint32_t tfull0 = empty0 + 8 * STAGES;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain = tempty0 + 16;
  const uint32_t ebar0 = drain + 8;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the pair MMAs
  const int pair = static_cast<int>(blockIdx.x) >> 1;
  const int npairs = static_cast<int>(gridDim.x) >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 2 * (EPI_THREADS / 32));  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    for (int i = 0; i < 16; ++i) mbar_init(ebar0 + 8 * i, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tma_a);
    tma_prefetch_desc(&tma_b);
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t full_even = mapa_shared(full0, 0);
  const uint32_t tempty_even = mapa_shared(tempty0, 0);

  const int ntiles = p.m_tiles * p.n_tiles;  // m_tiles counts 256-row pair tiles
  const int nunits = ntiles * p.splits;       // tiles x K-slices
  const uint32_t smem_base = smem_u32(smem);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int u = pair; u < nunits && ok; u += npairs) {
        int mt, nt;
        tile_coords(u % ntiles, p, mt, nt);
        const int m0 = (2 * mt + static_cast<int>(rank)) * BM;
        const int kb0 = (u / ntiles) * p.kb_split;
        const int kb1 = min(p.k_blocks, kb0 + p.kb_split);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, ph ^ 1, p.err)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(full0 + 8 * stage, 2 * STAGE_BYTES);
          const uint32_t fb = full_even + 8 * stage;
          const uint32_t sa = smem_base + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          const int k0 = kb * BK;
          if (A_MN) {
            tma_load_2d_pair(sa, &tma_a, fb, m0, k0);
            tma_load_2d_pair(sa + MN_CHUNK_BYTES, &tma_a, fb, m0 + 64, k0);
          } else {
            tma_load_2d_pair(sa, &tma_a, fb, k0, m0);
          }
          if (B_MN) {
            const int n0 = nt * BN + static_cast<int>(rank) * BH;
#pragma unroll
            for (int j = 0; j < BH / 64; ++j)
              tma_load_2d_pair(sb + j * MN_CHUNK_BYTES, &tma_b, fb, n0 + 64 * j, k0);
          } else {
            // one box of BN/2 rows; SwiGLU: the even CTA loads the 128 gate rows
            // of I-columns nt*128 + [0,128), the odd CTA the matching up rows
            const int r = (EPI == EPI_SWIGLU) ? nt * 128 + static_cast<int>(rank) * p.swiglu_half
                                              : nt * BN + static_cast<int>(rank) * BH;
            tma_load_2d_pair(sb, &tma_b, fb, k0, r);
          }
          if (++stage == STAGES) {
            stage = 0;
            ph ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ----------------------------------------------------------------- MMA
      constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN, A_MN, B_MN);
      const uint64_t a_desc0 = sdesc_sw128(smem_base, A_MN ? MN_CHUNK_BYTES : 16, 1024);
      const uint64_t b_desc0 = sdesc_sw128(smem_base + A_BYTES, B_MN ? MN_CHUNK_BYTES : 16, 1024);
      int stage = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t acc_ph = 0;
      bool ok = true;
      for (int u = pair; u < nunits && ok; u += npairs) {
        if (!mbar_wait_cluster(tempty0 + 8 * acc, acc_ph ^ 1, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        const int kb0 = (u / ntiles) * p.kb_split;
        const int kb1 = min(p.k_blocks, kb0 + p.kb_split);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, ph, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // descriptors of this stage: the ring's first stage plus the stage
          // offset, then one K=16 step = 32 B (K-major) or 2048 B (MN-major)
          const uint64_t ad0 = a_desc0 + static_cast<uint64_t>(stage) * (STAGE_BYTES >> 4);
          const uint64_t bd0 = b_desc0 + static_cast<uint64_t>(stage) * (STAGE_BYTES >> 4);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = ad0 + static_cast<uint64_t>(k) * ((A_MN ? 2048 : 32) >> 4);
            const uint64_t bd = bd0 + static_cast<uint64_t>(k) * ((B_MN ? 2048 : 32) >> 4);
            tc_mma_bf16_pair(d_tmem, ad, bd, idesc, kb != kb0 || k != 0);
          }
          tc_commit_pair_mc(empty0 + 8 * stage, 0x3);
          if (++stage == STAGES) {
            stage = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(tfull0 + 8 * acc, 0x3);
        acc ^= 1;
        if (acc == 0) acc_ph ^= 1;
      }
      // no pair MMA may still be writing either CTA's TMEM when it is released
      tc_commit_pair(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    uint8_t* stg = smem + TL::OFF_OUT + (warp - 2) * OS::BYTES;
    const Stage st{stg, smem_u32(stg), ebar0 + 16 * (warp - 2), lane};
    uint32_t ucnt = 0, eph = 0;
    int acc = 0;
    uint32_t acc_ph = 0;
    for (int u = pair; u < nunits; u += npairs) {
      int mt, nt;
      const int t = u % ntiles;
      tile_coords(t, p, mt, nt);
      const int mrow = 2 * mt + static_cast<int>(rank);
      const int row0 = (u / ntiles) * p.m_pad + mrow * BM + q * 32;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      if (!epilogue_tile<EPI, BN, OS::BYTES>(p, om, tbase, row0, nt, half, st,
                                             ucnt, eph, tfull0 + 8 * acc, acc_ph, t,
                                             static_cast<int>(rank) * 8 + (warp - 2)))
        break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_even + 8 * acc);
      acc ^= 1;
      if (acc == 0) acc_ph ^= 1;
    }
    if (lane == 0) bulk_wait0();
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync();
  if (p.err && *reinterpret_cast<volatile int*>(p.err) != 0) {
    // after a timed-out wait, copies issued just before may still be landing
    // on this pair's shared memory: let them finish before the CTAs exit
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 200000ull) {
    }
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------- host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

bool make_tma_2d(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld,
                 int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool make_map(CUtensorMap* m, const Mat& x, int box_rows) {
  return make_tma_2d(m, x.ptr, x.rows, x.cols, x.ld, box_rows);
}

// Map of an epilogue operand [rows, cols] (row stride ld elements, fp32 or
// bf16) with 32-row boxes of `unit` columns and the swizzle that matches the
// box's row bytes (128/64/32 B; none for 16 B), as stg_off lays them out.
static bool make_box_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld,
                         bool f32, int unit) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const int es = f32 ? 4 : 2;
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) || (ld * es) % 16) return false;
  const int rb = unit * es;
  const CUtensorMapSwizzle sw = rb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : rb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                : rb == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                           : CU_TENSOR_MAP_SWIZZLE_NONE;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * es};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(unit), 32u};
  cuuint32_t estr[2] = {1u, 1u};
  return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
             const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The maps an epilogue stores through and loads from (see OutMaps), for
// staging buffers of `stg` bytes per warp.
static bool make_out_maps(OutMaps* om, const Epi& e, int M, int N, uint32_t stg) {
  memset(om, 0, sizeof(*om));
  const int u = epi_unit(e.kind, stg);
  bf16* out = static_cast<bf16*>(e.out);
  switch (e.kind) {
    case EPI_F32:
      return make_box_map(&om->o1, e.out, M, N, e.ld_out, true, u);
    case EPI_F32_RESID:
      return make_box_map(&om->o1, e.out, M, N, e.ld_out, true, u) &&
             make_box_map(&om->i1, e.resid, M, N, e.ld_resid, true, u);
    case EPI_BF16:
    case EPI_CE_GRAD:
      return make_box_map(&om->o1, e.out, M, N, e.ld_out, false, u);
    case EPI_CE:
      return true;  // statistics only
    case EPI_SWIGLU:
      return make_box_map(&om->o1, out, M, e.half, e.ld_out, false, u) &&
             make_box_map(&om->o2, out + e.half, M, e.half, e.ld_out, false, u) &&
             make_box_map(&om->o3, e.out2, M, e.half, e.ld_out2, false, u);
    case EPI_SWIGLU_BWD:
      return make_box_map(&om->o1, out, M, N, e.ld_out, false, u) &&
             make_box_map(&om->o2, out + e.half, M, N, e.ld_out, false, u) &&
             make_box_map(&om->i1, e.aux, M, N, e.ld_aux, false, u) &&
             make_box_map(&om->i2, e.aux + e.half, M, N, e.ld_aux, false, u);
    default:
      return false;
  }
}

// Multiply-add FLOPs of one launch: 2 M N K, where the SwiGLU epilogue's
// N counts one half of the [gate | up] columns the tiles compute.
template <int EPI>
static double launch_flops(const GemmParams& p) {
  return 2.0 * p.M * static_cast<double>(p.N) * p.K * (EPI == EPI_SWIGLU ? 2.0 : 1.0);
}

template <int A_MN, int B_MN, int EPI, int BN>
static cudaError_t launch(const CUtensorMap& ta, const CUtensorMap& tb, const OutMaps& om,
                          const GemmParams& p, cudaStream_t s, bool timed = true) {
  static bool attr_done = false;  // per instantiation; the attribute is per function
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<A_MN, B_MN, EPI, BN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Tile<BN>::SMEM));
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int nunits = p.m_tiles * p.n_tiles * p.splits;
  const int grid = nunits < num_sms() ? nunits : num_sms();
  const int64_t slot = timed ? gemm_timing_before(s, launch_flops<EPI>(p), GEMM_KIND_SINGLE) : -1;
  note_launch();
  gemm_kernel<A_MN, B_MN, EPI, BN><<<grid, GEMM_THREADS, Tile<BN>::SMEM, s>>>(ta, tb, om, p);
  gemm_timing_after(s, slot);
  return cudaGetLastError();
}

template <int A_MN, int B_MN, int EPI, int BN>
static cudaError_t launch2(const CUtensorMap& ta, const CUtensorMap& tb, const OutMaps& om,
                           const GemmParams& p, int max_pairs, cudaStream_t s,
                           bool timed = true) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(gemm2_kernel<A_MN, B_MN, EPI, BN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Tile2<BN>::SMEM));
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int nunits = p.m_tiles * p.n_tiles * p.splits;
  const int pairs = nunits < max_pairs ? nunits : max_pairs;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = Tile2<BN>::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int64_t slot = timed ? gemm_timing_before(s, launch_flops<EPI>(p), GEMM_KIND_PAIR) : -1;
  note_launch();
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm2_kernel<A_MN, B_MN, EPI, BN>, ta, tb, om, p);
  gemm_timing_after(s, slot);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// CTA pairs that can be resident at once (clusters of 2 with the pair
// kernel's shared memory); 0 if clusters cannot be launched.
static int max_active_pairs() {
  static int n = -1;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * num_sms(), 1, 1);
    cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = Tile2<256>::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int c = 0;
    if (cudaFuncSetAttribute(gemm2_kernel<0, 0, EPI_F32, 256>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Tile2<256>::SMEM)) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&c, gemm2_kernel<0, 0, EPI_F32, 256>, &cfg) != cudaSuccess)
      c = 0;
    cudaGetLastError();
    n = c;
  });
  return n;
}

// Rows of the A operand per raster group: all row tiles when A fits in the L2
// budget (B streams once), 1 when B does (A streams once), else as many row
// tiles as fit.
static int raster_group(int m_tiles, int n_tiles, int rows_per_tile, int cols_per_tile, int K) {
  constexpr double kL2Budget = 48.0 * 1024 * 1024;
  const double a_tile = static_cast<double>(rows_per_tile) * K * 2;
  const double b_tile = static_cast<double>(cols_per_tile) * K * 2;
  if (a_tile * m_tiles <= kL2Budget) return m_tiles;
  if (b_tile * n_tiles <= kL2Budget) return 1;
  const int g = static_cast<int>(kL2Budget / a_tile);
  return g < 1 ? 1 : (g > m_tiles ? m_tiles : g);
}

int64_t gemm_sq_slots_bound(int M, int N) {
  return static_cast<int64_t>((M + BM - 1) / BM) * ((N + 127) / 128) * 16;
}

// Sum of the split-K partials (fp32 slabs of m_pad x ldw, added in split
// order) with the F32, F32_RESID or BF16 epilogue, four columns per thread
// (N % 4 == 0; the host falls back to one); F32 / F32_RESID also write one fp64
// squared-sum slot per block (fixed grid and order: deterministic).
template <int V>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(
    const float* __restrict__ ws, int splits, int64_t slab, int64_t ldw, int M, int N, int kind,
    void* __restrict__ out, int64_t ld_out, float scale, const float* __restrict__ resid,
    int64_t ld_resid, double* __restrict__ sq_part) {
  __shared__ double red[8];
  double acc = 0.0;
  const int nv = N / V;
  const int64_t n = static_cast<int64_t>(M) * nv;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / nv;
    const int64_t c = (i - r * nv) * V;
    const float* w = ws + r * ldw + c;
    float v[V];
    if constexpr (V == 4) {
      const float4 a = *reinterpret_cast<const float4*>(w);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    } else {
      v[0] = w[0];
    }
    for (int sp = 1; sp < splits; ++sp) {
      if constexpr (V == 4) {
        const float4 a = *reinterpret_cast<const float4*>(w + sp * slab);
        v[0] += a.x; v[1] += a.y; v[2] += a.z; v[3] += a.w;
      } else {
        v[0] += w[sp * slab];
      }
    }
    if (kind == EPI_F32_RESID) {
      const float* rs = resid + r * ld_resid + c;
      if constexpr (V == 4) {
        const float4 a = *reinterpret_cast<const float4*>(rs);
        v[0] = a.x + v[0]; v[1] = a.y + v[1]; v[2] = a.z + v[2]; v[3] = a.w + v[3];
      } else {
        v[0] = rs[0] + v[0];
      }
    }
    if (kind == EPI_F32 || kind == EPI_F32_RESID) {
      float* o = static_cast<float*>(out) + r * ld_out + c;
      if constexpr (V == 4) *reinterpret_cast<float4*>(o) = make_float4(v[0], v[1], v[2], v[3]);
      else o[0] = v[0];
#pragma unroll
      for (int k = 0; k < V; ++k) acc += static_cast<double>(v[k]) * v[k];
    } else {
      bf16* o = static_cast<bf16*>(out) + r * ld_out + c;
      if constexpr (V == 4)
        *reinterpret_cast<uint2*>(o) =
            make_uint2(pack_bf16x2(scale * v[0], scale * v[1]), pack_bf16x2(scale * v[2], scale * v[3]));
      else
        o[0] = __float2bfloat16_rn(scale * v[0]);
    }
  }
  if (!sq_part) return;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < 8; ++w) t += red[w];
    sq_part[blockIdx.x] = t;
  }
}

// Launches splitk_reduce_kernel over partial slabs of m_pad x ldw in epi.split_ws.
static cudaError_t splitk_reduce(const Epi& epi, int splits, int64_t m_pad, int64_t ldw, int M,
                                 int N, cudaStream_t s) {
  // four columns per thread when every row stays 16 (fp32) / 8 (bf16) byte aligned
  const int es = epi.kind == EPI_BF16 ? 2 : 4;
  bool vec = N % 4 == 0 && epi.ld_out % 4 == 0 &&
             (reinterpret_cast<uintptr_t>(epi.out) % (4 * es)) == 0;
  if (epi.kind == EPI_F32_RESID)
    vec = vec && epi.ld_resid % 4 == 0 && (reinterpret_cast<uintptr_t>(epi.resid) % 16) == 0;
  const int64_t items = static_cast<int64_t>(M) * (vec ? N / 4 : N);
  const bool sq = (epi.kind == EPI_F32 || epi.kind == EPI_F32_RESID) && epi.sq_part;
  int64_t nblk = (items + 255) / 256;
  nblk = std::max<int64_t>(1, std::min<int64_t>(nblk, sq ? gemm_sq_slots_bound(M, N)
                                                         : 8LL * num_sms()));
  if (sq) *epi.sq_count = nblk;
  note_launch();
  if (vec)
    splitk_reduce_kernel<4><<<static_cast<unsigned>(nblk), 256, 0, s>>>(
        epi.split_ws, splits, m_pad * ldw, ldw, M, N, epi.kind, epi.out, epi.ld_out, epi.scale,
        epi.resid, epi.ld_resid, sq ? epi.sq_part : nullptr);
  else
    splitk_reduce_kernel<1><<<static_cast<unsigned>(nblk), 256, 0, s>>>(
        epi.split_ws, splits, m_pad * ldw, ldw, M, N, epi.kind, epi.out, epi.ld_out, epi.scale,
        epi.resid, epi.ld_resid, sq ? epi.sq_part : nullptr);
  return cudaGetLastError();
}

// C = A' B'^T as `splits` K-slices on single-CTA 128 x 256 tiles whose fp32
// partials go to epi.split_ws, then splitk_reduce_kernel.
static cudaError_t gemm_splitk(const Mat& A, bool a_mn, const Mat& B, bool b_mn, int M, int N,
                               int K, int splits, const Epi& epi, int* err, cudaStream_t s,
                               const char** why) {
  const int kbs = (K + BK - 1) / BK;
  const int kb_split = (kbs + splits - 1) / splits;
  splits = (kbs + kb_split - 1) / kb_split;  // no empty slice
  const int m_tiles = (M + BM - 1) / BM;
  const int64_t m_pad = static_cast<int64_t>(m_tiles) * BM;
  const int64_t ldw = (N + 3) / 4 * 4;
  Epi pe;
  pe.kind = EPI_F32;
  pe.out = epi.split_ws;
  pe.ld_out = ldw;
  CUtensorMap ta, tb;
  if (!make_map(&ta, A, a_mn ? 64 : 128) || !make_map(&tb, B, 64)) {
    *why = "gemm: cuTensorMapEncodeTiled failed";
    return cudaErrorInvalidValue;
  }
  OutMaps om;
  if (!make_out_maps(&om, pe, static_cast<int>(splits * m_pad), N, OutStageBytes(256))) {
    *why = "gemm: split-K scratch needs 16-byte alignment";
    return cudaErrorInvalidValue;
  }
  GemmParams p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.m_tiles = m_tiles;
  p.n_tiles = (N + 255) / 256;
  p.k_blocks = kbs;
  p.swiglu_half = 0;
  p.group = raster_group(p.m_tiles, p.n_tiles, BM, 256, K);
  p.sq_slots = 8;
  p.kb_main = kbs;
  p.splits = splits;
  p.kb_split = kb_split;
  p.m_pad = static_cast<int>(m_pad);
  p.m_epi = static_cast<int>(splits * m_pad);
  p.epi = pe;
  p.err = err;
  cudaError_t e = cudaErrorInvalidValue;
  // the timed interval covers the K-slices and their reduce
  const int64_t slot = gemm_timing_before(s, launch_flops<EPI_F32>(p), GEMM_KIND_SINGLE);
  if (!a_mn && !b_mn) e = launch<0, 0, EPI_F32, 256>(ta, tb, om, p, s, false);
  else if (!a_mn && b_mn) e = launch<0, 1, EPI_F32, 256>(ta, tb, om, p, s, false);
  else if (a_mn && b_mn) e = launch<1, 1, EPI_F32, 256>(ta, tb, om, p, s, false);
  else *why = "gemm: unsupported operand-major combination for split-K";
  if (e == cudaSuccess) e = splitk_reduce(epi, splits, m_pad, ldw, M, N, s);
  gemm_timing_after(s, slot);
  return e;
}

// C = A' B'^T as `splits` K-slices on CTA-pair 256 x 256 tiles whose fp32
// partials go to epi.split_ws, then splitk_reduce_kernel.
static cudaError_t gemm_splitk_pair(const Mat& A, bool a_mn, const Mat& B, bool b_mn, int M, int N,
                                    int K, int splits, int pairs_max, const Epi& epi, int* err,
                                    cudaStream_t s, const char** why) {
  const int kbs = (K + BK - 1) / BK;
  const int kb_split = (kbs + splits - 1) / splits;
  splits = (kbs + kb_split - 1) / kb_split;  // no empty slice
  const int m_tiles = (M + 2 * BM - 1) / (2 * BM);
  const int64_t m_pad = static_cast<int64_t>(m_tiles) * 2 * BM;
  const int64_t ldw = (N + 3) / 4 * 4;
  Epi pe;
  pe.kind = EPI_F32;
  pe.out = epi.split_ws;
  pe.ld_out = ldw;
  CUtensorMap ta, tb;
  if (!make_map(&ta, A, a_mn ? 64 : 128) || !make_map(&tb, B, b_mn ? 64 : 128)) {
    *why = "gemm: cuTensorMapEncodeTiled failed";
    return cudaErrorInvalidValue;
  }
  OutMaps om;
  if (!make_out_maps(&om, pe, static_cast<int>(splits * m_pad), N, OutStageBytes(256))) {
    *why = "gemm: split-K scratch needs 16-byte alignment";
    return cudaErrorInvalidValue;
  }
  GemmParams p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.m_tiles = m_tiles;
  p.n_tiles = (N + 255) / 256;
  p.k_blocks = kbs;
  p.swiglu_half = 0;
  p.group = raster_group(p.m_tiles, p.n_tiles, 2 * BM, 256, K);
  p.sq_slots = 16;
  p.kb_main = kbs;
  p.splits = splits;
  p.kb_split = kb_split;
  p.m_pad = static_cast<int>(m_pad);
  p.m_epi = static_cast<int>(splits * m_pad);
  p.epi = pe;
  p.err = err;
  cudaError_t e = cudaErrorInvalidValue;
  // the timed interval covers the K-slices and their reduce
  const int64_t slot = gemm_timing_before(s, launch_flops<EPI_F32>(p), GEMM_KIND_PAIR);
  if (!a_mn && !b_mn) e = launch2<0, 0, EPI_F32, 256>(ta, tb, om, p, pairs_max, s, false);
  else if (!a_mn && b_mn) e = launch2<0, 1, EPI_F32, 256>(ta, tb, om, p, pairs_max, s, false);
  else if (a_mn && b_mn) e = launch2<1, 1, EPI_F32, 256>(ta, tb, om, p, pairs_max, s, false);
  else *why = "gemm: unsupported operand-major combination for split-K";
  if (e == cudaSuccess) e = splitk_reduce(epi, splits, m_pad, ldw, M, N, s);
  gemm_timing_after(s, slot);
  return e;
}

cudaError_t gemm(const Mat& A, bool a_mn, const Mat& B, bool b_mn, int M, int N, int K,
                 const Epi& epi, int* err, cudaStream_t s, const char** why) {
  if (M <= 0 || N <= 0 || K <= 0) {
    *why = "gemm: empty problem";
    return cudaErrorInvalidValue;
  }
  const bool swiglu = epi.kind == EPI_SWIGLU;
  if (swiglu && b_mn) {
    *why = "gemm: SwiGLU epilogue needs a K-major B";
    return cudaErrorInvalidValue;
  }
  if ((A.ld % 8) || (B.ld % 8) || (reinterpret_cast<uintptr_t>(A.ptr) & 15) ||
      (reinterpret_cast<uintptr_t>(B.ptr) & 15)) {
    *why = "gemm: operands need 16-byte aligned rows";
    return cudaErrorInvalidValue;
  }
  // Tile shape: single-CTA 128 x 256 or 128 x 192, or CTA-pair 256 x 256.
  // Cost = waves x per-CTA tile width / mainloop rate, with the rates of the
  // three shapes measured on the projection and LM-head GEMMs of a Qwen3-4B
  // step (pair 1.05, single 256 1.0, single 192 0.85): the pair mainloop
  // moves a third fewer bytes per flop; 192-wide tiles win where they cut a
  // wave (N = 2560 outputs).
  constexpr double kRate256 = 1.0, kRate192 = 0.85, kRatePair = 1.05;
  const bool fixed256 = swiglu || epi.kind == EPI_CE;
  const int sms = num_sms();
  const int pairs_max = max_active_pairs();
  auto cost1 = [&](int w, double rate) {
    const int64_t tiles = (int64_t)((M + BM - 1) / BM) * ((N + w - 1) / w);
    return static_cast<double>((tiles + sms - 1) / sms) * w / rate;
  };
  bool pair_tiles = false;
  int bn = 256;
  double best = cost1(256, kRate256);
  if (!fixed256 && cost1(192, kRate192) < best) {
    best = cost1(192, kRate192);
    bn = 192;
  }
  if (pairs_max > 0 && M > BM) {
    auto cost2 = [&](int w, double rate) {
      const int64_t tiles = (int64_t)((M + 2 * BM - 1) / (2 * BM)) * ((N + w - 1) / w);
      return static_cast<double>((tiles + pairs_max - 1) / pairs_max) * w / rate;
    };
    if (cost2(256, kRatePair) < best) {
      best = cost2(256, kRatePair);
      bn = 256;
      pair_tiles = true;
    }
  }
  if (epi.split_ws && (epi.kind == EPI_F32 || epi.kind == EPI_F32_RESID || epi.kind == EPI_BF16)) {
    const int64_t tiles1 = (int64_t)((M + BM - 1) / BM) * ((N + 255) / 256);
    const int kbs = (K + BK - 1) / BK;
    const int64_t m_pad = (int64_t)((M + BM - 1) / BM) * BM;
    const int64_t ldw = (N + 3) / 4 * 4;
    int64_t splits = std::min<int64_t>(sms / tiles1, kbs / 4);
    while (splits > 1 && splits * m_pad * ldw > epi.split_ws_floats) --splits;
    if (splits >= 2)
      return gemm_splitk(A, a_mn, B, b_mn, M, N, K, static_cast<int>(splits), epi, err, s, why);
  }
  // K-slices for CTA-pair tiles that would leave much of a wave idle (the
  // N = 2560 outputs of a 4096-token step: 160 tiles on 76 pairs): estimated
  // time = rounds of work units x one slice's share of a pair-tile (about
  // 1.6 PFLOP/s over the pairs) + the partials' round trip through memory.
  if (pair_tiles && epi.split_ws && (epi.kind == EPI_F32 || epi.kind == EPI_F32_RESID)) {
    const int64_t tiles = static_cast<int64_t>((M + 2 * BM - 1) / (2 * BM)) * ((N + 255) / 256);
    const int64_t m_pad = static_cast<int64_t>((M + 2 * BM - 1) / (2 * BM)) * 2 * BM;
    const int64_t ldw = (N + 3) / 4 * 4;
    const int kbs = (K + BK - 1) / BK;
    const double tile_us = 2.0 * 256 * 256 * K * pairs_max / 1.6e15 * 1e6;
    auto cost = [&](int sl) {
      double c = static_cast<double>((tiles * sl + pairs_max - 1) / pairs_max) * tile_us / sl;
      if (sl > 1) c += (sl + 2) * static_cast<double>(M) * N * 4 / 5.0e12 * 1e6 + 3.0;
      return c;
    };
    int bs = 1;
    double bc = cost(1);
    for (int sl = 2; sl <= 4; ++sl) {
      if (sl * m_pad * ldw > epi.split_ws_floats || kbs < 4 * sl) break;
      if (cost(sl) < 0.97 * bc) {
        bc = cost(sl);
        bs = sl;
      }
    }
    if (bs > 1)
      return gemm_splitk_pair(A, a_mn, B, b_mn, M, N, K, bs, pairs_max, epi, err, s, why);
  }
  CUtensorMap ta, tb;
  const int b_box = (pair_tiles && !b_mn) ? bn / 2 : 64;
  if (!make_map(&ta, A, a_mn ? 64 : 128) || !make_map(&tb, B, b_box)) {
    *why = "gemm: cuTensorMapEncodeTiled failed";
    return cudaErrorInvalidValue;
  }
  OutMaps om;
  if (!make_out_maps(&om, epi, M, N, OutStageBytes(bn))) {
    *why = "gemm: outputs need 16-byte aligned rows (cuTensorMapEncodeTiled failed)";
    return cudaErrorInvalidValue;
  }
  GemmParams p;
  p.M = M;
  p.N = N;
  p.K = K;
  const int rows_per_tile = pair_tiles ? 2 * BM : BM;
  p.m_tiles = (M + rows_per_tile - 1) / rows_per_tile;
  p.n_tiles = swiglu ? (N + 127) / 128 : (N + bn - 1) / bn;
  p.k_blocks = (K + BK - 1) / BK;
  p.swiglu_half = epi.half;
  p.group = raster_group(p.m_tiles, p.n_tiles, rows_per_tile, swiglu ? 256 : bn, K);
  p.sq_slots = pair_tiles ? 16 : 8;
  p.splits = 1;
  p.kb_split = p.k_blocks;
  p.m_pad = p.m_tiles * rows_per_tile;
  p.m_epi = M;
  p.epi = epi;
  p.epi.sq_count = nullptr;
  p.err = err;
  if (epi.sq_part) {
    if ((epi.kind != EPI_F32 && epi.kind != EPI_F32_RESID) || !epi.sq_count) {
      *why = "gemm: squared-sum slots need an fp32 epilogue and a count";
      return cudaErrorInvalidValue;
    }
    *epi.sq_count = static_cast<int64_t>(p.m_tiles) * p.n_tiles * p.sq_slots;
  }
#define RDT_GEMM_CASE(AM, BMJ, E, W)                                           \
  if (!pair_tiles && a_mn == (AM) && b_mn == (BMJ) && epi.kind == (E) && bn == (W)) \
    return launch<AM, BMJ, E, W>(ta, tb, om, p, s);
#define RDT_GEMM2_CASE(AM, BMJ, E, W)                                          \
  if (pair_tiles && a_mn == (AM) && b_mn == (BMJ) && epi.kind == (E) && bn == (W)) \
    return launch2<AM, BMJ, E, W>(ta, tb, om, p, pairs_max, s);
  // forward projections: A K-major, B K-major
  RDT_GEMM_CASE(0, 0, EPI_BF16, 256)
  RDT_GEMM_CASE(0, 0, EPI_BF16, 192)
  RDT_GEMM_CASE(0, 0, EPI_F32, 256)
  RDT_GEMM_CASE(0, 0, EPI_F32, 192)
  RDT_GEMM_CASE(0, 0, EPI_F32_RESID, 256)
  RDT_GEMM_CASE(0, 0, EPI_F32_RESID, 192)
  RDT_GEMM_CASE(0, 0, EPI_SWIGLU, 256)
  RDT_GEMM_CASE(0, 0, EPI_CE, 256)
  RDT_GEMM2_CASE(0, 0, EPI_BF16, 256)
  RDT_GEMM2_CASE(0, 0, EPI_F32, 256)
  RDT_GEMM2_CASE(0, 0, EPI_F32_RESID, 256)
  RDT_GEMM2_CASE(0, 0, EPI_SWIGLU, 256)
  RDT_GEMM2_CASE(0, 0, EPI_CE, 256)
  RDT_GEMM_CASE(0, 0, EPI_CE_GRAD, 256)
  RDT_GEMM_CASE(0, 0, EPI_CE_GRAD, 192)
  RDT_GEMM2_CASE(0, 0, EPI_CE_GRAD, 256)
  // activation gradients dX = dY W: A K-major, B MN-major
  RDT_GEMM_CASE(0, 1, EPI_BF16, 256)
  RDT_GEMM_CASE(0, 1, EPI_BF16, 192)
  RDT_GEMM_CASE(0, 1, EPI_F32, 256)
  RDT_GEMM_CASE(0, 1, EPI_F32, 192)
  RDT_GEMM_CASE(0, 1, EPI_F32_RESID, 256)  // the LM head's dh, summed over vocabulary chunks
  RDT_GEMM_CASE(0, 1, EPI_F32_RESID, 192)
  RDT_GEMM_CASE(0, 1, EPI_SWIGLU_BWD, 256)
  RDT_GEMM_CASE(0, 1, EPI_SWIGLU_BWD, 192)
  RDT_GEMM2_CASE(0, 1, EPI_BF16, 256)
  RDT_GEMM2_CASE(0, 1, EPI_F32, 256)
  RDT_GEMM2_CASE(0, 1, EPI_F32_RESID, 256)
  RDT_GEMM2_CASE(0, 1, EPI_SWIGLU_BWD, 256)
  // weight gradients dW = dY^T X: A MN-major, B MN-major
  RDT_GEMM_CASE(1, 1, EPI_F32, 256)
  RDT_GEMM_CASE(1, 1, EPI_F32, 192)
  RDT_GEMM_CASE(1, 1, EPI_F32_RESID, 256)  // gradient accumulation: dW += dY^T X
  RDT_GEMM_CASE(1, 1, EPI_F32_RESID, 192)
  RDT_GEMM_CASE(1, 1, EPI_BF16, 256)
  RDT_GEMM_CASE(1, 1, EPI_BF16, 192)
  RDT_GEMM2_CASE(1, 1, EPI_F32, 256)
  RDT_GEMM2_CASE(1, 1, EPI_F32_RESID, 256)
  RDT_GEMM2_CASE(1, 1, EPI_BF16, 256)
#undef RDT_GEMM2_CASE
#undef RDT_GEMM_CASE
  *why = "gemm: unsupported operand-major / epilogue combination";
  return cudaErrorInvalidValue;
}

// ------------------------------------------------------------- NF4 host
static bool make_u8_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols_bytes,
                        int box_cols, int box_rows, CUtensorMapSwizzle sw) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || (reinterpret_cast<uintptr_t>(ptr) & 15) || (cols_bytes % 16)) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols_bytes), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols_bytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
static bool make_f32_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols,
                         int box_cols, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || (reinterpret_cast<uintptr_t>(ptr) & 15) || ((cols * 4) % 16)) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int B_MN, int EPI>
static cudaError_t launch_nf4_pair(const CUtensorMap& ta, const CUtensorMap& tb2,
                                   const Nf4Maps& nm, const OutMaps& om, const GemmParams& p,
                                   int max_pairs, cudaStream_t s, bool timed = true) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(gemm2_nf4_kernel<B_MN, EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(TileN4P::SMEM));
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int nunits = p.m_tiles * p.n_tiles * p.splits;
  const int pairs = nunits < max_pairs ? nunits : max_pairs;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(NF4P_THREADS, 1, 1);
  cfg.dynamicSmemBytes = TileN4P::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int64_t slot = timed ? gemm_timing_before(s, launch_flops<EPI>(p), GEMM_KIND_NF4) : -1;
  note_launch();
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm2_nf4_kernel<B_MN, EPI>, ta, tb2, nm, om, p);
  gemm_timing_after(s, slot);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// CTA pairs of the NF4 pair kernel that can be resident at once (0: none).
static int max_active_nf4_pairs() {
  static int n = -1;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * num_sms(), 1, 1);
    cfg.blockDim = dim3(NF4P_THREADS, 1, 1);
    cfg.dynamicSmemBytes = TileN4P::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int c = 0;
    if (cudaFuncSetAttribute(gemm2_nf4_kernel<0, EPI_F32>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(TileN4P::SMEM)) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&c, gemm2_nf4_kernel<0, EPI_F32>, &cfg) != cudaSuccess)
      c = 0;
    cudaGetLastError();
    n = c;
  });
  return n;
}

template <int B_MN, int EPI>
static cudaError_t launch_nf4(const CUtensorMap& ta, const CUtensorMap& tb2, const Nf4Maps& nm,
                              const OutMaps& om, const GemmParams& p, cudaStream_t s,
                              bool timed = true) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(gemm_nf4_kernel<B_MN, EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(TileN4::SMEM));
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int ntiles = p.m_tiles * p.n_tiles;
  const int grid = ntiles < num_sms() ? ntiles : num_sms();
  const int64_t slot = timed ? gemm_timing_before(s, launch_flops<EPI>(p), GEMM_KIND_NF4) : -1;
  note_launch();
  gemm_nf4_kernel<B_MN, EPI><<<grid, NF4_THREADS, TileN4::SMEM, s>>>(ta, tb2, nm, om, p);
  gemm_timing_after(s, slot);
  return cudaGetLastError();
}

cudaError_t gemm_nf4(const Mat& A, const Nf4Mat& W, bool b_mn, const Mat* A2, const Mat* B2,
                     int K2, int M, const Epi& epi, int* err, cudaStream_t s, const char** why) {
  const bool swiglu = epi.kind == EPI_SWIGLU;
  // SwiGLU: W is the stacked [Wg; Wu] and N the width of one half
  const int N = static_cast<int>(b_mn ? W.cols : (swiglu ? W.rows / 2 : W.rows));
  const int K1 = static_cast<int>(b_mn ? W.rows : W.cols);
  if (swiglu && (epi.half != N || W.rows != 2 * static_cast<int64_t>(N) || N % 128)) {
    *why = "gemm_nf4: SwiGLU needs W = [Wg; Wu] with half = rows / 2, a multiple of 128";
    return cudaErrorInvalidValue;
  }
  if (M <= 0 || N <= 0 || K1 <= 0 || K2 < 0 || K2 > BK) {
    *why = "gemm_nf4: empty problem or a tail wider than 64";
    return cudaErrorInvalidValue;
  }
  if (W.cols % 256 || W.rows % 64 || (K2 > 0 && (!A2 || !B2))) {
    *why = "gemm_nf4: NF4 weights need cols % 256 == 0 and rows % 64 == 0";
    return cudaErrorInvalidValue;
  }
  if (swiglu && b_mn) {
    *why = "gemm_nf4: SwiGLU epilogue needs a K-major B";
    return cudaErrorInvalidValue;
  }
  if ((A.ld % 8) || (reinterpret_cast<uintptr_t>(A.ptr) & 15) ||
      (K2 > 0 && ((A2->ld % 8) || (B2->ld % 8) || (reinterpret_cast<uintptr_t>(A2->ptr) & 15) ||
                  (reinterpret_cast<uintptr_t>(B2->ptr) & 15)))) {
    *why = "gemm_nf4: operands need 16-byte aligned rows";
    return cudaErrorInvalidValue;
  }
  // CTA pairs whenever there are two 128-row halves to pair (and clusters launch)
  const int pairs_max = max_active_nf4_pairs();
  const bool pair_tiles = pairs_max > 0 && M > BM;
  CUtensorMap ta, tb2;
  Nf4Maps nm;
  bool ok = make_map(&ta, A, 128);
  // MN-major code rows (128 bytes per CTA, 64 per CTA of a pair) swizzled so
  // the decode warps' reads spread over the banks
  const CUtensorMapSwizzle csw = !b_mn        ? CU_TENSOR_MAP_SWIZZLE_NONE
                                 : pair_tiles ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_128B;
  ok = ok && make_u8_map(&nm.codes, W.codes, W.rows, W.cols / 2,
                         b_mn ? (pair_tiles ? 64 : 128) : 32, 64, csw);
  ok = ok && make_f32_map(&nm.scales, W.scales, W.rows, W.cols / 64, 4, 64);
  if (K2 > 0) {
    ok = ok && make_map(&nm.a2, *A2, 128) && make_map(&tb2, *B2, 64);
  } else {
    nm.a2 = ta;
    tb2 = ta;
  }
  if (!ok) {
    *why = "gemm_nf4: cuTensorMapEncodeTiled failed";
    return cudaErrorInvalidValue;
  }
  OutMaps om;
  if (!make_out_maps(&om, epi, M, N, OutStageBytes(NF4_BN))) {
    *why = "gemm_nf4: outputs need 16-byte aligned rows";
    return cudaErrorInvalidValue;
  }
  GemmParams p;
  p.M = M;
  p.N = N;
  p.K = K1 + K2;
  const int rows_per_tile = pair_tiles ? 2 * BM : BM;
  p.m_tiles = (M + rows_per_tile - 1) / rows_per_tile;
  p.n_tiles = swiglu ? (N + 127) / 128 : (N + NF4_BN - 1) / NF4_BN;
  p.kb_main = K1 / BK;
  p.k_blocks = p.kb_main + (K2 > 0 ? 1 : 0);
  p.swiglu_half = epi.half;
  p.group = raster_group(p.m_tiles, p.n_tiles, rows_per_tile, swiglu ? 256 : NF4_BN, p.K);
  p.sq_slots = pair_tiles ? 16 : 8;
  p.splits = 1;
  p.kb_split = p.k_blocks;
  p.m_pad = p.m_tiles * rows_per_tile;
  p.m_epi = M;
  p.epi = epi;
  p.epi.sq_count = nullptr;
  p.err = err;
  if (epi.sq_part) {
    if (epi.kind != EPI_F32 || !epi.sq_count) {
      *why = "gemm_nf4: squared-sum slots need the fp32 epilogue and a count";
      return cudaErrorInvalidValue;
    }
    *epi.sq_count = static_cast<int64_t>(p.m_tiles) * p.n_tiles * p.sq_slots;
  }
  // K-slices for pair tiles that would leave most of a wave idle (the N = 2560
  // outputs of a 2048-token step: 80 tiles on 76 pairs). Estimated time =
  // rounds of work units x one slice's share of a tile (a pair-tile at about
  // 1 PFLOP/s over the pairs) + the partials' round trip through memory; the
  // fp32 partials are then summed in slice order with the epilogue applied.
  if (pair_tiles && (epi.kind == EPI_F32 || epi.kind == EPI_F32_RESID) && !epi.sq_part &&
      epi.split_ws) {
    const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
    const int64_t m_pad = static_cast<int64_t>(p.m_tiles) * 2 * BM;
    const int64_t ldw = (N + 3) / 4 * 4;
    const double tile_us = 2.0 * 256 * 256 * p.K * pairs_max / 1.0e15 * 1e6;
    auto cost = [&](int sl) {
      const double rounds = static_cast<double>((tiles * sl + pairs_max - 1) / pairs_max);
      double c = rounds * tile_us / sl;
      if (sl > 1) c += (sl + 2) * static_cast<double>(M) * N * 4 / 5.0e12 * 1e6 + 3.0;
      return c;
    };
    int best = 1;
    double best_cost = cost(1);
    for (int sl = 2; sl <= 4; ++sl) {
      if (sl * m_pad * ldw > epi.split_ws_floats || p.k_blocks < 4 * sl) break;
      const double c = cost(sl);
      if (c < 0.97 * best_cost) {
        best_cost = c;
        best = sl;
      }
    }
    if (best > 1) {
      Epi pe;
      pe.kind = EPI_F32;
      pe.out = epi.split_ws;
      pe.ld_out = ldw;
      OutMaps oms;
      p.kb_split = (p.k_blocks + best - 1) / best;
      p.splits = (p.k_blocks + p.kb_split - 1) / p.kb_split;  // no empty slice
      p.m_pad = static_cast<int>(m_pad);
      p.m_epi = static_cast<int>(p.splits * m_pad);
      if (!make_out_maps(&oms, pe, p.m_epi, N, OutStageBytes(NF4_BN))) {
        *why = "gemm_nf4: split-K scratch needs 16-byte alignment";
        return cudaErrorInvalidValue;
      }
      p.epi = pe;
      // the timed interval covers the K-slices and their reduce
      const int64_t slot = gemm_timing_before(s, launch_flops<EPI_F32>(p), GEMM_KIND_NF4);
      cudaError_t e =
          b_mn ? launch_nf4_pair<1, EPI_F32>(ta, tb2, nm, oms, p, pairs_max, s, false)
               : launch_nf4_pair<0, EPI_F32>(ta, tb2, nm, oms, p, pairs_max, s, false);
      if (e == cudaSuccess) e = splitk_reduce(epi, p.splits, m_pad, ldw, M, N, s);
      gemm_timing_after(s, slot);
      return e;
    }
  }
#define RDT_NF4_CASE(BMJ, E)                                                   \
  if (b_mn == (BMJ) && epi.kind == (E))                                        \
    return pair_tiles ? launch_nf4_pair<BMJ, E>(ta, tb2, nm, om, p, pairs_max, s) \
                      : launch_nf4<BMJ, E>(ta, tb2, nm, om, p, s);
  // forward through W: y = x W^T (K-major)
  RDT_NF4_CASE(0, EPI_F32)
  RDT_NF4_CASE(0, EPI_F32_RESID)
  RDT_NF4_CASE(0, EPI_SWIGLU)
  // activation gradients through W: dX = dY W (MN-major)
  RDT_NF4_CASE(1, EPI_F32)
  RDT_NF4_CASE(1, EPI_BF16)
  RDT_NF4_CASE(1, EPI_SWIGLU_BWD)
#undef RDT_NF4_CASE
  *why = "gemm_nf4: unsupported operand-major / epilogue combination";
  return cudaErrorInvalidValue;
}

}  // namespace rdt
