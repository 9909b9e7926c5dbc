// Internal host-side interface between the C-ABI layer and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rdt {

using bf16 = __nv_bfloat16;

// Epilogue applied to each 128 x 256 fp32 accumulator tile of the GEMM.
enum EpiKind : int {
  EPI_BF16 = 0,        // out(bf16)[r, c] = acc
  EPI_F32 = 1,         // out(f32)[r, c] = acc
  EPI_F32_RESID = 2,   // out(f32)[r, c] = resid[r, c] + acc
  EPI_SWIGLU = 3,      // B = [Wg; Wu]: gu[r, c] = g, gu[r, half + c] = u, out2[r, c] = silu(g) u
  EPI_SWIGLU_BWD = 4,  // acc = ds: out[r, c] = dg, out[r, half + c] = du from aux = gu
  // acc = logits of vocabulary columns col_off + c:
  EPI_CE = 5,       // part[r, 2*tile+half] = (max, sum exp), tgt_logit[r] if the target is here
  EPI_CE_GRAD = 6,  // out(bf16) = scale * (exp(z - lse[r]) - [col_off + c == targets[r]])
};

struct Epi {
  int kind = EPI_F32;
  void* out = nullptr;
  int64_t ld_out = 0;
  const float* resid = nullptr;
  int64_t ld_resid = 0;
  void* out2 = nullptr;
  int64_t ld_out2 = 0;
  const bf16* aux = nullptr;
  int64_t ld_aux = 0;
  int half = 0;
  float2* part = nullptr;
  int part_ld = 0;
  const int32_t* targets = nullptr;
  float* tgt_logit = nullptr;
  // EPI_F32 / EPI_F32_RESID: when set, every epilogue warp writes the fp64
  // sum of the squares of the values it stored, one slot per (tile, warp),
  // and the host gemm() sets *sq_count to the number of slots written (tiles
  // x 8 or 16; or the split-K reduce's blocks).
  double* sq_part = nullptr;
  int64_t* sq_count = nullptr;
  // EPI_BF16: out = bf16(scale * acc); EPI_CE_GRAD: the loss scale
  float scale = 1.0f;
  // EPI_CE_GRAD: per-row log-sum-exp; EPI_CE / EPI_CE_GRAD: vocabulary index of column 0
  const float* lse = nullptr;
  int col_off = 0;
  // F32 / F32_RESID / BF16: fp32 scratch gemm() may use to split K across CTAs when the
  // problem has too few output tiles to fill the GPU (split_ws_floats floats,
  // 16-byte aligned); the partials are summed in a fixed order.
  float* split_ws = nullptr;
  int64_t split_ws_floats = 0;
};

// Upper bound of the squared-sum slots a gemm() of [M, N] writes.
int64_t gemm_sq_slots_bound(int M, int N);

// A bf16 row-major matrix in global memory.
struct Mat {
  const void* ptr;
  int64_t rows, cols, ld;
};

// C[M, N] = A' B'^T over K, where
//   A' = A        ([M, K], K contiguous) when !a_mn, else A^T with A given as [K, M];
//   B' = B        ([N, K], K contiguous) when !b_mn, else B^T with B given as [K, N].
// For EPI_SWIGLU, B is the stacked [2*half, K] matrix and N = half.
// Returns cudaSuccess or an error; on a host-side rejection *why is set.
cudaError_t gemm(const Mat& A, bool a_mn, const Mat& B, bool b_mn, int M, int N, int K,
                 const Epi& epi, int* err, cudaStream_t s, const char** why);

// A frozen NF4 weight W [rows, cols] (row-major, two 4-bit codes per byte,
// element 2j in the low nibble of byte j; one fp32 scale per 64 consecutive
// elements of a row; cols % 256 == 0).
struct Nf4Mat {
  const uint8_t* codes;
  const float* scales;
  int64_t rows, cols;
};

// C[M, N] = A' B'^T with B decoded from NF4 on the way: !b_mn: B = W (N =
// rows, K = cols; y = x W^T); b_mn: B = W^T (N = cols, K = rows; dX = dY W).
// A is K-major bf16 [M, K]. K2 > 0 (<= 64) appends a tail of ordinary bf16
// operands: A2 [M, K2] K-major and B2 ([N, K2] K-major when !b_mn, [K2, N]
// MN-major when b_mn). Epilogues as gemm() (F32, F32_RESID, SWIGLU forward;
// F32, BF16, SWIGLU_BWD backward).
cudaError_t gemm_nf4(const Mat& A, const Nf4Mat& W, bool b_mn, const Mat* A2, const Mat* B2,
                     int K2, int M, const Epi& epi, int* err, cudaStream_t s, const char** why);

// (max, sum exp) partials per row written by the CE epilogue: one per half of
// every 256-wide N tile.
inline int ce_partials_per_row(int N) { return 2 * ((N + 255) / 256); }

int num_sms();

// 2-D bf16 TMA map over a row-major [rows, cols] matrix (row stride ld
// elements) with a box of 64 columns x box_rows rows and 128-byte swizzle.
bool make_tma_2d(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld,
                 int box_rows);

// Sets the thread-local message returned by rdt_last_error().
void set_last_error(const char* msg);

// Kernel-launch bookkeeping (librdt-wide): every launch site calls note_launch.
void note_launch(int n = 1);
// GEMM timing hook: called around each GEMM launch (see rdt_gemm_timing_arm).
// kind: GEMM_KIND_SINGLE (one CTA per tile), GEMM_KIND_PAIR (CTA pair),
// GEMM_KIND_NF4 (NF4-decoding kernel).
enum GemmKind : int { GEMM_KIND_SINGLE = 0, GEMM_KIND_PAIR = 1, GEMM_KIND_NF4 = 2 };
int64_t gemm_timing_before(cudaStream_t s, double flops, int kind);
void gemm_timing_after(cudaStream_t s, int64_t slot);

// Upper bound on the row count of any gain-gradient partials buffer.
constexpr int kMaxPartialRows = 512;
// Upper bound on the per-block partials of the squared sum.
constexpr int kMaxSqSumPartials = 4096;

// ------------------------------------------------------------ elementwise
cudaError_t rmsnorm_fwd(const float* x, const float* gamma, bf16* y, float* rstd, int T, int H,
                        float eps, cudaStream_t s);
// dx = rstd*(dy*g - xhat*mean(dy*g*xhat)) + resid (resid may be null);
// dx_bf16 optional; dgamma partials [nblk, H] then reduced into dgamma
// (dgamma = sum, or dgamma += sum when accumulate).
cudaError_t rmsnorm_bwd(const float* dy, const float* x, const float* rstd, const float* gamma,
                        const float* resid, float* dx, bf16* dx_bf16, float* dgamma,
                        float* partials, int T, int H, cudaStream_t s, bool accumulate = false);
int rmsnorm_bwd_partial_rows(int T, int threads);

cudaError_t rope_table(float* cs, int S, int d, float theta, cudaStream_t s);
// qkv: fp32 raw projections [T, ld] (q | k | v); writes the normalised and
// rotated q, k and a bf16 copy of v.
cudaError_t qknorm_rope_fwd(const float* qkv, int64_t ld_qkv, bf16* q_out, bf16* k_out,
                            bf16* v_out, float* rstd_q, float* rstd_k, const float* gq,
                            const float* gk, const float* cs, int T, int S, int nh, int nkv, int d,
                            float eps, cudaStream_t s);
// dg_qk: 2*d floats, q-gain gradient then k-gain gradient (= or += when
// accumulate).
cudaError_t qknorm_rope_bwd(const float* dq, const float* dk, const float* qkv, int64_t ld_qkv,
                            const float* rstd_q, const float* rstd_k, const float* gq,
                            const float* gk, const float* cs, bf16* dqkv, float* dg_qk,
                            float* partials, int T, int S, int nh, int nkv, int d,
                            cudaStream_t s, bool accumulate = false);
int qknorm_bwd_partial_rows(int T, int heads);

// *out (= or +=, per `accumulate`) the fp64 sum of parts[0, n) plus the sums
// of squares of up to 4 small fp32 arrays, in a fixed order: kSqCtas CTAs
// write slice sums to scratch[kSqCtas], one warp adds them in index order.
constexpr int kSqCtas = 64;
cudaError_t sq_reduce(const double* parts, int64_t n, const float* const* small,
                      const int64_t* small_len, int nsmall, double* out, bool accumulate,
                      double* scratch, cudaStream_t s);
// out [sum of rows, np*r] bf16, block diagonal: rows of piece p (fp32
// [rows_p, r], row-major) land in columns [p r, (p+1) r), zeros elsewhere.
cudaError_t lora_bstack(const float* const* pieces, const int64_t* rows, int np, int r,
                        bf16* out, cudaStream_t s);
cudaError_t cast_bf16(const float* src, bf16* dst, int64_t n, cudaStream_t s);

// ---------------------------------------------------------------- embedding
cudaError_t embedding_forward(const float* table, int64_t V, int H, const int32_t* ids, int T,
                              float* x, int* err, cudaStream_t s);
size_t embedding_workspace_bytes(int T);
cudaError_t embedding_backward(const int32_t* ids, int T, const float* dx, int H,
                               const float* scale, float* dtable, int64_t V, bool accumulate,
                               void* ws, cudaStream_t s);

// Folds one vocabulary chunk's per-tile (max, sum exp) partials [T, part_ld]
// (ntiles used) into the running per-row statistics run[T]; the first chunk
// starts them, the last writes lse[T] and loss[T] = lse - tgt_logit.
cudaError_t ce_merge(const float2* part, int part_ld, int ntiles, float2* run, bool first,
                     bool last, const float* tgt_logit, float* lse, float* loss, int T,
                     cudaStream_t s);

// One-warp kernel that waits on an mbarrier with limit_ns (arrived on first
// when `arrive`), holding and then freeing 32 TMEM columns; a wait that gives
// up records the timeout code in *err. waited_ns (device, nullable) receives
// the wait's duration.
cudaError_t wait_probe(int* err, uint64_t limit_ns, bool arrive, unsigned long long* waited_ns,
                       cudaStream_t s);

cudaError_t sq_sum(const float* const* bufs, const int64_t* lens, int nbuf, double* out,
                   double* partials, int max_partials, cudaStream_t s);
cudaError_t clip_scale(const double* sumsq, float max_norm, float* scale, int32_t* nonfinite,
                       cudaStream_t s);
cudaError_t adamw(float* w, const float* g, float* m, float* v, int64_t n, const float* scale,
                  const int32_t* skip, float lr, float b1, float b2, float eps, float wd,
                  float bc1, float bc2, bf16* wb, cudaStream_t s,
                  const int32_t* step_dev = nullptr);
// *step += 1 on the device (the optimizer's step count, read by adamw when
// its step lives on the device, e.g. under graph replay).
cudaError_t step_advance(int32_t* step, cudaStream_t s);

// ---------------------------------------------------------------- attention
// mma.sync flash attention (attention.cu) for head_dim 16 and 32.
// q [T, ldq] (head h at column h*d), k/v [T, ldk/ldv] (kv head g at g*d),
// o [T, nh*d] bf16, lse [B, nh, S] fp32 (natural log).
cudaError_t attn_fwd(const bf16* q, int64_t ldq, const bf16* k, int64_t ldk, const bf16* v,
                     int64_t ldv, bf16* o, float* lse, int B, int S, int nh, int nkv, int d,
                     cudaStream_t s);
// D[(b*nh + h)*S_ld + s] = sum_d dO * O; if lse2 != null also
// lse2[same] = lse[(b*nh + h)*S + s] * log2(e); 0 in both for S <= s < S_ld.
// d in {16, 32, 64, 128}.
cudaError_t attn_bwd_pre(const bf16* o, const bf16* dout, const float* lse, float* D,
                         float* lse2, int B, int S, int S_ld, int nh, int d, cudaStream_t s);
// Row stride (>= S, multiple of 64) of the D / lse2 arrays the tensor-core backward reads.
int attn_lse_pad(int S);
// dq (fp32 [T, nh*d], must be zeroed; accumulated), dk fp32 [T, nkv*d],
// dv bf16 written at dv + t*lddv + g*d.
cudaError_t attn_bwd(const bf16* q, int64_t ldq, const bf16* k, int64_t ldk, const bf16* v,
                     int64_t ldv, const bf16* dout, const float* lse, const float* D, float* dq,
                     float* dk, bf16* dv, int64_t lddv, int B, int S, int nh, int nkv, int d,
                     cudaStream_t s);

// tcgen05 flash attention (attention_tc.cu): forward and backward for
// head_dim 64/128; same arguments as attn_fwd / attn_bwd plus the
// device error word for bounded waits. The backward reads lse2 (log2-domain
// LSE) and D in the padded [B*nh, attn_lse_pad(S)] layout and writes every
// dq element (no zeroing needed).
bool attn_tc_supported(int d, bool backward);
cudaError_t attn_fwd_tc(const bf16* q, int64_t ldq, const bf16* k, int64_t ldk, const bf16* v,
                        int64_t ldv, bf16* o, float* lse, int B, int S, int nh, int nkv, int d,
                        int* err, cudaStream_t s);
cudaError_t attn_bwd_tc(const bf16* q, int64_t ldq, const bf16* k, int64_t ldk, const bf16* v,
                        int64_t ldv, const bf16* dout, const float* lse, const float* D,
                        float* dq, float* dk, bf16* dv, int64_t lddv, int B, int S, int nh,
                        int nkv, int d, int* err, cudaStream_t s);

}  // namespace rdt
