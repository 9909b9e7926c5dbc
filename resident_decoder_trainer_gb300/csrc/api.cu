// C-ABI entry points of librdt.so (declared in include/rdt.h): argument
// validation, carving of the caller's saved-activation and scratch buffers,
// and the launch sequence of each call. Nothing here allocates device memory.
#include <cmath>
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>

#include "../../include/rdt.h"
#include "internal.h"

using namespace rdt;

namespace {

thread_local std::string g_last_error;

rdt_status fail(rdt_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

// Device error word: bounded waits that give up record a code here.
__device__ int g_device_error;

int* device_error_ptr() {
  static int* ptrs[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

// ---------------------------------------------------------- measurement hooks
std::atomic<int64_t> g_launches{0};
std::mutex g_timing_mu;
void* const* g_timing_events = nullptr;
double* g_timing_flops = nullptr;
int32_t* g_timing_kinds = nullptr;
int32_t g_timing_cap = 0;
int64_t g_timing_seen = 0;
bool g_timing_armed = false;

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Sequential carve of a caller buffer into 256-byte aligned pieces.
struct Carver {
  uint8_t* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<uint8_t*>(b)) {}
  template <typename T>
  T* take(size_t count) {
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off = align_up(off + count * sizeof(T));
    return p;
  }
};

bool cfg_ok(const rdt_config* c, std::string* why) {
  if (!c) { *why = "config is null"; return false; }
  if (c->hidden < 16 || c->hidden > 4096 || c->hidden % 16) {
    *why = "hidden must be a multiple of 16 in [16, 4096]"; return false;
  }
  if (!(c->head_dim == 16 || c->head_dim == 32 || c->head_dim == 64 || c->head_dim == 128)) {
    *why = "head_dim must be 16, 32, 64 or 128"; return false;
  }
  if (c->n_heads < 1 || c->n_kv_heads < 1 || c->n_heads % c->n_kv_heads) {
    *why = "n_heads must be a positive multiple of n_kv_heads"; return false;
  }
  if (c->intermediate < 16 || c->intermediate % 16) {
    *why = "intermediate must be a positive multiple of 16"; return false;
  }
  if (c->vocab < 16 || c->vocab % 16) { *why = "vocab must be a positive multiple of 16"; return false; }
  if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) {
    *why = "rms_eps must be >= 0 and rope_theta > 0"; return false;
  }
  return true;
}

struct Dims {
  int64_t H, nh, nkv, d, I, V, qd, kd, nqkv;
};
Dims dims_of(const rdt_config* c) {
  Dims m;
  m.H = c->hidden; m.nh = c->n_heads; m.nkv = c->n_kv_heads; m.d = c->head_dim;
  m.I = c->intermediate; m.V = c->vocab;
  m.qd = m.nh * m.d; m.kd = m.nkv * m.d; m.nqkv = m.qd + 2 * m.kd;
  return m;
}

void block_counts(const Dims& m, int64_t* cnt) {
  cnt[RDT_WQ] = m.qd * m.H;
  cnt[RDT_WK] = m.kd * m.H;
  cnt[RDT_WV] = m.kd * m.H;
  cnt[RDT_WO] = m.H * m.qd;
  cnt[RDT_WG] = m.I * m.H;
  cnt[RDT_WU] = m.I * m.H;
  cnt[RDT_WD] = m.H * m.I;
  cnt[RDT_G_ATTN] = m.H;
  cnt[RDT_G_FFN] = m.H;
  cnt[RDT_G_Q] = m.d;
  cnt[RDT_G_K] = m.d;
}
void block_offsets(const Dims& m, int64_t* off) {
  int64_t cnt[RDT_BLOCK_NTENSORS];
  block_counts(m, cnt);
  int64_t o = 0;
  for (int i = 0; i < RDT_BLOCK_NTENSORS; ++i) {
    off[i] = o;
    o += cnt[i];  // every count is a multiple of 16
  }
}

// Saved activations of one block.
struct Saved {
  bf16 *xn, *vb, *qr, *kr, *o, *xn2, *gu, *s;
  float *qkv, *rstd1, *rstd_q, *rstd_k, *lse, *r1, *rstd2;
};
size_t carve_saved(const Dims& m, int64_t B, int64_t S, void* base, Saved* sv) {
  const int64_t T = B * S;
  Carver c(base);
  Saved t;
  t.xn = c.take<bf16>(T * m.H);
  t.rstd1 = c.take<float>(T);
  t.qkv = c.take<float>(T * m.nqkv);  // raw projections, fp32 (QK-norm input)
  t.vb = c.take<bf16>(T * m.kd);      // v as the attention operand
  t.qr = c.take<bf16>(T * m.qd);
  t.kr = c.take<bf16>(T * m.kd);
  t.rstd_q = c.take<float>(T * m.nh);
  t.rstd_k = c.take<float>(T * m.nkv);
  t.o = c.take<bf16>(T * m.qd);
  t.lse = c.take<float>(B * m.nh * S);
  t.r1 = c.take<float>(T * m.H);
  t.xn2 = c.take<bf16>(T * m.H);
  t.rstd2 = c.take<float>(T);
  t.gu = c.take<bf16>(T * 2 * m.I);
  t.s = c.take<bf16>(T * m.I);
  if (sv) *sv = t;
  return c.off;
}

// Scratch of block forward / backward (one layout serves both).
struct BlockWs {
  float* cs;
  bf16 *dy_b, *dgu, *dr1_b, *dout, *dqkv;
  float *dxn, *dr1, *Dd, *lse2, *dq, *dk, *partials;
  double* sqp;  // squared-sum slots of the weight-gradient GEMMs
  double* sq2;  // their per-CTA partial sums (kSqCtas)
  float* split;  // split-K partials of the [T, hidden] projections
  int64_t split_floats;
};
// fp32 scratch for four K-slices of a [T, H] GEMM output on 256-row tiles
inline int64_t split_floats_for(int64_t T, int64_t H) { return 4 * ((T + 255) / 256 * 256) * H; }
size_t carve_block_ws(const Dims& m, int64_t B, int64_t S, void* base, BlockWs* w) {
  const int64_t T = B * S;
  Carver c(base);
  BlockWs t;
  t.cs = c.take<float>(S * m.d);  // [S][d/2] (cos, sin)
  t.dy_b = c.take<bf16>(T * m.H);
  t.dgu = c.take<bf16>(T * 2 * m.I);
  t.dr1_b = c.take<bf16>(T * m.H);
  t.dout = c.take<bf16>(T * m.qd);
  t.dqkv = c.take<bf16>(T * m.nqkv);
  t.dxn = c.take<float>(T * m.H);
  t.dr1 = c.take<float>(T * m.H);
  t.Dd = c.take<float>(B * m.nh * attn_lse_pad((int)S));
  t.lse2 = c.take<float>(B * m.nh * attn_lse_pad((int)S));
  t.dq = c.take<float>(T * m.qd);
  t.dk = c.take<float>(T * m.kd);
  const int64_t pw = m.H > 2 * m.d ? m.H : 2 * m.d;
  t.partials = c.take<float>(kMaxPartialRows * pw);
  t.sqp = c.take<double>(gemm_sq_slots_bound((int)m.H, (int)m.I) +
                         gemm_sq_slots_bound((int)(2 * m.I), (int)m.H) +
                         gemm_sq_slots_bound((int)m.H, (int)m.qd) +
                         gemm_sq_slots_bound((int)m.nqkv, (int)m.H));
  t.sq2 = c.take<double>(kSqCtas);
  t.split_floats = split_floats_for(T, m.H);
  t.split = c.take<float>(t.split_floats);
  if (w) *w = t;
  return c.off;
}

// Vocabulary columns per chunk of the LM head: the chunk's bf16 dz [T, Vc]
// holds at most 128 M elements (256 MB; the whole vocabulary if smaller), a
// fixed bound whatever V is. Fewer, larger chunks run faster than chunks that
// stay in L2 (one Qwen3-4B head step, 4096 tokens: 8.1 ms at 64 MB, 7.65 ms
// at 128 MB, 7.26 ms at 256 MB), through fewer launches and fuller waves of
// the dW_lm GEMM.
int64_t ce_chunk_cols(int64_t T, int64_t V) {
  int64_t vc = ((int64_t)128 << 20) / T / 256 * 256;
  if (vc < 256) vc = 256;
  return vc < V ? vc : V;
}

struct HeadWs {
  bf16 *hn, *dz;
  float *rstd, *tgt, *lse, *dhn, *partials;
  float2 *part, *run;
  int64_t vc;    // vocabulary columns per chunk
  int part_ld;   // (max, sum exp) partials per row of one chunk
  double* sqp;   // squared-sum slots of the dW_lm GEMMs
  double* sq2;   // their per-CTA partial sums (kSqCtas)
  float* split;  // split-K partials of dh_n
  int64_t split_floats;
};
size_t carve_head_ws(const Dims& m, int64_t T, void* base, HeadWs* w) {
  Carver c(base);
  HeadWs t;
  t.vc = ce_chunk_cols(T, m.V);
  t.part_ld = ce_partials_per_row((int)t.vc);
  t.hn = c.take<bf16>(T * m.H);
  t.rstd = c.take<float>(T);
  t.dz = c.take<bf16>(T * t.vc);
  t.part = c.take<float2>(T * t.part_ld);
  t.run = c.take<float2>(T);
  t.tgt = c.take<float>(T);
  t.lse = c.take<float>(T);
  t.dhn = c.take<float>(T * m.H);
  t.partials = c.take<float>(kMaxPartialRows * m.H);
  int64_t slots = 0;
  for (int64_t v0 = 0; v0 < m.V; v0 += t.vc)
    slots += gemm_sq_slots_bound((int)std::min(t.vc, m.V - v0), (int)m.H);
  t.sqp = c.take<double>(slots);
  t.sq2 = c.take<double>(kSqCtas);
  t.split_floats = split_floats_for(T, m.H);
  t.split = c.take<float>(t.split_floats);
  if (w) *w = t;
  return c.off;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

#define RDT_CHECK_CUDA(expr)                                                     \
  do {                                                                           \
    cudaError_t e_ = (expr);                                                     \
    if (e_ != cudaSuccess)                                                       \
      return fail(RDT_ECUDA, "%s failed: %s", #expr, cudaGetErrorString(e_));    \
  } while (0)

#define RDT_GEMM(...)                                                                 \
  do {                                                                                \
    const char* why_ = "";                                                           \
    cudaError_t e_ = gemm(__VA_ARGS__, &why_);                                        \
    if (e_ != cudaSuccess)                                                            \
      return fail(*why_ ? RDT_EINVAL : RDT_ECUDA, "gemm at line %d: %s %s", __LINE__, \
                  why_, cudaGetErrorString(e_));                                      \
  } while (0)

#define RDT_GEMM_NF4(...)                                                             \
  do {                                                                                \
    const char* why_ = "";                                                           \
    cudaError_t e_ = gemm_nf4(__VA_ARGS__, &why_);                                    \
    if (e_ != cudaSuccess)                                                            \
      return fail(*why_ ? RDT_EINVAL : RDT_ECUDA, "nf4 gemm at line %d: %s %s",        \
                  __LINE__, why_, cudaGetErrorString(e_));                            \
  } while (0)

}  // namespace

namespace rdt {
void set_last_error(const char* msg) { g_last_error = msg ? msg : ""; }

void note_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int64_t gemm_timing_before(cudaStream_t s, double flops, int kind) {
  std::lock_guard<std::mutex> lk(g_timing_mu);
  if (!g_timing_armed) return -1;
  const int64_t slot = g_timing_seen++;
  if (slot >= g_timing_cap) return -1;
  g_timing_flops[slot] = flops;
  if (g_timing_kinds) g_timing_kinds[slot] = kind;
  cudaEventRecord(static_cast<cudaEvent_t>(g_timing_events[2 * slot]), s);
  return slot;
}

void gemm_timing_after(cudaStream_t s, int64_t slot) {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lk(g_timing_mu);
  if (g_timing_armed && slot < g_timing_cap)
    cudaEventRecord(static_cast<cudaEvent_t>(g_timing_events[2 * slot + 1]), s);
}
}  // namespace rdt

// ------------------------------------------------------- NF4 + LoRA layout
namespace {

bool nf4_ok(const rdt_config* c, int rank, std::string* why) {
  if (!cfg_ok(c, why)) return false;
  const Dims m = dims_of(c);
  if (m.H % 256 || m.qd % 256 || m.I % 256) {
    *why = "NF4: hidden, n_heads*head_dim and intermediate must be multiples of 256";
    return false;
  }
  if (m.kd % 64) {
    *why = "NF4: n_kv_heads*head_dim must be a multiple of 64";
    return false;
  }
  if (rank != 8 && rank != 16) {
    *why = "NF4: LoRA rank must be 8 or 16";
    return false;
  }
  return true;
}

// Projections in storage order: q, k, v, o, gate, up, down as [out, in].
void nf4_dims(const Dims& m, int64_t* out, int64_t* in) {
  const int64_t o[7] = {m.qd, m.kd, m.kd, m.H, m.I, m.I, m.H};
  const int64_t i[7] = {m.H, m.H, m.H, m.qd, m.H, m.H, m.I};
  for (int k = 0; k < 7; ++k) {
    out[k] = o[k];
    in[k] = i[k];
  }
}
void nf4_layout(const Dims& m, int64_t* code_off, int64_t* scale_off, int64_t* code_total,
                int64_t* scale_total) {
  int64_t out[7], in[7];
  nf4_dims(m, out, in);
  int64_t c = 0, sc = 0;
  for (int k = 0; k < 7; ++k) {
    if (code_off) code_off[k] = c;
    if (scale_off) scale_off[k] = sc;
    c += out[k] * in[k] / 2;
    sc += out[k] * in[k] / 64;
  }
  if (code_total) *code_total = c;
  if (scale_total) *scale_total = sc;
}
void lora_layout(const Dims& m, int64_t r, int64_t* off, int64_t* cnt) {
  int64_t out[7], in[7];
  nf4_dims(m, out, in);
  int64_t c[RDT_LORA_NTENSORS];
  for (int k = 0; k < 7; ++k) {
    c[RDT_LORA_A_Q + k] = r * in[k];
    c[RDT_LORA_B_Q + k] = out[k] * r;
  }
  int64_t o = 0;
  for (int k = 0; k < RDT_LORA_NTENSORS; ++k) {
    if (off) off[k] = o;
    if (cnt) cnt[k] = c[k];
    o += c[k];
  }
}
// Shadow (bf16): the A's as in the adapter layout, then the B stacks:
// [Bq; Bk; Bv] block diagonal [nqkv, 3r], Bo [H, r], [Bg; Bu] block diagonal
// [2I, 2r], Bd [H, r].
struct LoraShadow {
  const bf16 *a_qkv, *a_o, *a_gu, *a_d, *b_qkv, *b_o, *b_gu, *b_d;
  int64_t total;
};
LoraShadow lora_shadow_layout(const Dims& m, int64_t r, const bf16* base) {
  int64_t off[RDT_LORA_NTENSORS], cnt[RDT_LORA_NTENSORS];
  lora_layout(m, r, off, cnt);
  const int64_t a_end = off[RDT_LORA_B_Q];
  LoraShadow t;
  t.a_qkv = base + off[RDT_LORA_A_Q];
  t.a_o = base + off[RDT_LORA_A_O];
  t.a_gu = base + off[RDT_LORA_A_G];
  t.a_d = base + off[RDT_LORA_A_D];
  int64_t o = a_end;
  t.b_qkv = base + o;
  o += m.nqkv * 3 * r;
  t.b_o = base + o;
  o += m.H * r;
  t.b_gu = base + o;
  o += 2 * m.I * 2 * r;
  t.b_d = base + o;
  o += m.H * r;
  t.total = o;
  return t;
}

// Saved by the NF4 forward beyond the block's: the scaled down-projections
// U = s x A^T of the four GEMM inputs (bf16 [T, 3r], [T, r], [T, 2r], [T, r]).
struct Nf4Saved {
  bf16 *u_qkv, *u_o, *u_gu, *u_d;
};
size_t carve_nf4_saved(const Dims& m, int64_t r, int64_t B, int64_t S, void* base, Saved* sv,
                       Nf4Saved* nv) {
  const size_t head = carve_saved(m, B, S, base, sv);
  const int64_t T = B * S;
  Carver c(base ? static_cast<uint8_t*>(base) + head : nullptr);
  Nf4Saved t;
  t.u_qkv = c.take<bf16>(T * 3 * r);
  t.u_o = c.take<bf16>(T * r);
  t.u_gu = c.take<bf16>(T * 2 * r);
  t.u_d = c.take<bf16>(T * r);
  if (nv) *nv = t;
  return head + c.off;
}
// Scratch of the NF4 backward beyond the block's: dU = s dY B per GEMM and
// sinks for the frozen gains' gradients.
struct Nf4Ws {
  bf16 *du_qkv, *du_o, *du_gu, *du_d;
  float* gain_sink;
  double* sqp;  // squared-sum slots of the adapter-gradient GEMMs
  double* sq2;  // their per-CTA partial sums (kSqCtas)
  float* split;  // split-K partials of the adapter GEMMs (few output tiles, long K)
  int64_t split_floats;
};
// Squared-sum slots the fourteen adapter-gradient GEMMs write at most.
int64_t lora_sq_slots_bound(const Dims& m, int64_t r) {
  const int R = (int)r;
  return gemm_sq_slots_bound((int)m.H, R) + gemm_sq_slots_bound(R, (int)m.I) +
         2 * gemm_sq_slots_bound((int)m.I, R) + gemm_sq_slots_bound(2 * R, (int)m.H) +
         gemm_sq_slots_bound((int)m.H, R) + gemm_sq_slots_bound(R, (int)m.qd) +
         gemm_sq_slots_bound((int)m.qd, R) + 2 * gemm_sq_slots_bound((int)m.kd, R) +
         gemm_sq_slots_bound(3 * R, (int)m.H);
}
size_t carve_nf4_ws(const Dims& m, int64_t r, int64_t B, int64_t S, void* base, BlockWs* wk,
                    Nf4Ws* nw) {
  const size_t head = carve_block_ws(m, B, S, base, wk);
  const int64_t T = B * S;
  Carver c(base ? static_cast<uint8_t*>(base) + head : nullptr);
  Nf4Ws t;
  t.du_qkv = c.take<bf16>(T * 3 * r);
  t.du_o = c.take<bf16>(T * r);
  t.du_gu = c.take<bf16>(T * 2 * r);
  t.du_d = c.take<bf16>(T * r);
  t.gain_sink = c.take<float>(2 * m.H + 2 * m.d);
  t.sqp = c.take<double>(lora_sq_slots_bound(m, r));
  t.sq2 = c.take<double>(kSqCtas);
  // room for 8 K-slices of the widest [r..3r, out] adapter gradient, 16 of
  // the [T, 3r] down-projections
  const int64_t wide = std::max(std::max(m.H, m.I), std::max(m.qd, m.nqkv));
  const int64_t t_pad = (T + 127) / 128 * 128;
  // ... or 4 of the [T, hidden] outputs of the NF4 projections (256-row pair tiles)
  const int64_t t_pad2 = (T + 255) / 256 * 256;
  t.split_floats = std::max<int64_t>(std::max<int64_t>(8 * 128 * wide, 16 * t_pad * 3 * r),
                                     4 * t_pad2 * m.H);
  t.split = c.take<float>(t.split_floats);
  if (nw) *nw = t;
  return head + c.off;
}

}  // namespace

// =========================================================================
extern "C" {

rdt_status rdt_gemm_timing_arm(void* const* events, double* flops, int32_t* kinds,
                               int32_t capacity) {
  if (!events || !flops || capacity < 1) return fail(RDT_EINVAL, "events/flops/capacity");
  std::lock_guard<std::mutex> lk(g_timing_mu);
  g_timing_events = events;
  g_timing_flops = flops;
  g_timing_kinds = kinds;
  g_timing_cap = capacity;
  g_timing_seen = 0;
  g_timing_armed = true;
  return RDT_OK;
}

int64_t rdt_gemm_timing_disarm(void) {
  std::lock_guard<std::mutex> lk(g_timing_mu);
  g_timing_armed = false;
  g_timing_events = nullptr;
  g_timing_flops = nullptr;
  g_timing_kinds = nullptr;
  return g_timing_seen;
}

int64_t rdt_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* rdt_last_error(void) { return g_last_error.c_str(); }

rdt_status rdt_check_config(const rdt_config* cfg) {
  std::string why;
  if (!cfg_ok(cfg, &why)) return fail(RDT_EINVAL, "config: %s", why.c_str());
  return RDT_OK;
}

int64_t rdt_block_param_count(const rdt_config* cfg) {
  std::string why;
  if (!cfg_ok(cfg, &why)) return -1;
  int64_t cnt[RDT_BLOCK_NTENSORS];
  block_counts(dims_of(cfg), cnt);
  int64_t s = 0;
  for (int i = 0; i < RDT_BLOCK_NTENSORS; ++i) s += cnt[i];
  return s;
}

rdt_status rdt_block_param_offsets(const rdt_config* cfg, int64_t* offsets, int64_t* counts) {
  std::string why;
  if (!cfg_ok(cfg, &why)) return fail(RDT_EINVAL, "config: %s", why.c_str());
  if (!offsets || !counts) return fail(RDT_EINVAL, "offsets/counts is null");
  const Dims m = dims_of(cfg);
  block_offsets(m, offsets);
  block_counts(m, counts);
  return RDT_OK;
}

size_t rdt_block_saved_bytes(const rdt_config* cfg, int32_t batch, int32_t seq) {
  std::string why;
  if (!cfg_ok(cfg, &why) || batch < 1 || seq < 1) return 0;
  return carve_saved(dims_of(cfg), batch, seq, nullptr, nullptr);
}

size_t rdt_block_workspace_bytes(const rdt_config* cfg, int32_t batch, int32_t seq) {
  std::string why;
  if (!cfg_ok(cfg, &why) || batch < 1 || seq < 1) return 0;
  return carve_block_ws(dims_of(cfg), batch, seq, nullptr, nullptr);
}

size_t rdt_head_workspace_bytes(const rdt_config* cfg, int32_t tokens) {
  std::string why;
  if (!cfg_ok(cfg, &why) || tokens < 1) return 0;
  return carve_head_ws(dims_of(cfg), tokens, nullptr, nullptr);
}

size_t rdt_sq_sum_workspace_bytes(void) { return kMaxSqSumPartials * sizeof(double); }

// -------------------------------------------------------------- block fwd
rdt_status rdt_block_forward(const rdt_config* cfg, int32_t batch, int32_t seq, const float* w,
                             const rdt_bf16* w_bf16, const float* x, float* y, void* saved,
                             size_t saved_bytes, void* ws, size_t ws_bytes, void* stream) {
  std::string why;
  if (!cfg_ok(cfg, &why)) return fail(RDT_EINVAL, "config: %s", why.c_str());
  if (batch < 1 || seq < 1) return fail(RDT_EINVAL, "batch and seq must be >= 1");
  if (!w || !w_bf16 || !x || !y || !saved || !ws) return fail(RDT_EINVAL, "null pointer");
  if (!aligned16(w) || !aligned16(w_bf16) || !aligned16(x) || !aligned16(y) ||
      (reinterpret_cast<uintptr_t>(saved) & 255) || (reinterpret_cast<uintptr_t>(ws) & 255))
    return fail(RDT_EINVAL, "w/x/y must be 16-byte and saved/ws 256-byte aligned");
  if (x == y) return fail(RDT_EINVAL, "y must not alias x");
  const Dims m = dims_of(cfg);
  if (saved_bytes < carve_saved(m, batch, seq, nullptr, nullptr))
    return fail(RDT_EINVAL, "saved buffer too small");
  if (ws_bytes < carve_block_ws(m, batch, seq, nullptr, nullptr))
    return fail(RDT_EINVAL, "workspace too small");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = device_error_ptr();
  const int T = batch * seq;
  Saved sv;
  carve_saved(m, batch, seq, saved, &sv);
  BlockWs wk;
  carve_block_ws(m, batch, seq, ws, &wk);
  int64_t off[RDT_BLOCK_NTENSORS];
  block_offsets(m, off);
  const bf16* wb = reinterpret_cast<const bf16*>(w_bf16);

  // input RMSNorm
  RDT_CHECK_CUDA(rmsnorm_fwd(x, w + off[RDT_G_ATTN], sv.xn, sv.rstd1, T, (int)m.H, cfg->rms_eps, s));
  // stacked Q/K/V projection: qkv[T, qd+2kd] = xn [Wq; Wk; Wv]^T (fp32)
  {
    Epi e;
    e.kind = EPI_F32;
    e.out = sv.qkv;
    e.ld_out = m.nqkv;
    RDT_GEMM(Mat{sv.xn, T, m.H, m.H}, false, Mat{wb + off[RDT_WQ], m.nqkv, m.H, m.H}, false, T,
             (int)m.nqkv, (int)m.H, e, err, s);
  }
  // per-head QK RMSNorm + RoPE-neox
  RDT_CHECK_CUDA(rope_table(wk.cs, seq, (int)m.d, cfg->rope_theta, s));
  RDT_CHECK_CUDA(qknorm_rope_fwd(sv.qkv, m.nqkv, sv.qr, sv.kr, sv.vb, sv.rstd_q, sv.rstd_k,
                                 w + off[RDT_G_Q], w + off[RDT_G_K], wk.cs, T, seq, (int)m.nh,
                                 (int)m.nkv, (int)m.d, cfg->rms_eps, s));
  // causal GQA attention
  if (attn_tc_supported((int)m.d, false))
    RDT_CHECK_CUDA(attn_fwd_tc(sv.qr, m.qd, sv.kr, m.kd, sv.vb, m.kd, sv.o,
                               sv.lse, batch, seq, (int)m.nh, (int)m.nkv, (int)m.d, err, s));
  else
    RDT_CHECK_CUDA(attn_fwd(sv.qr, m.qd, sv.kr, m.kd, sv.vb, m.kd, sv.o, sv.lse,
                            batch, seq, (int)m.nh, (int)m.nkv, (int)m.d, s));
  // O projection + residual: r1 = x + o Wo^T
  {
    Epi e;
    e.kind = EPI_F32_RESID;
    e.out = sv.r1;
    e.ld_out = m.H;
    e.resid = x;
    e.ld_resid = m.H;
    e.split_ws = wk.split;
    e.split_ws_floats = wk.split_floats;
    RDT_GEMM(Mat{sv.o, T, m.qd, m.qd}, false, Mat{wb + off[RDT_WO], m.H, m.qd, m.qd}, false, T,
             (int)m.H, (int)m.qd, e, err, s);
  }
  // post-attention RMSNorm
  RDT_CHECK_CUDA(rmsnorm_fwd(sv.r1, w + off[RDT_G_FFN], sv.xn2, sv.rstd2, T, (int)m.H,
                             cfg->rms_eps, s));
  // gate/up projection with the SwiGLU epilogue
  {
    Epi e;
    e.kind = EPI_SWIGLU;
    e.out = sv.gu;
    e.ld_out = 2 * m.I;
    e.out2 = sv.s;
    e.ld_out2 = m.I;
    e.half = (int)m.I;
    RDT_GEMM(Mat{sv.xn2, T, m.H, m.H}, false, Mat{wb + off[RDT_WG], 2 * m.I, m.H, m.H}, false, T,
             (int)m.I, (int)m.H, e, err, s);
  }
  // down projection + residual: y = r1 + s Wd^T
  {
    Epi e;
    e.kind = EPI_F32_RESID;
    e.out = y;
    e.ld_out = m.H;
    e.resid = sv.r1;
    e.ld_resid = m.H;
    e.split_ws = wk.split;
    e.split_ws_floats = wk.split_floats;
    RDT_GEMM(Mat{sv.s, T, m.I, m.I}, false, Mat{wb + off[RDT_WD], m.H, m.I, m.I}, false, T,
             (int)m.H, (int)m.I, e, err, s);
  }
  return RDT_OK;
}

// ------------------------------------------------------------- block bwd
rdt_status rdt_block_backward(const rdt_config* cfg, int32_t batch, int32_t seq, const float* w,
                              const rdt_bf16* w_bf16, const float* x, const void* saved,
                              size_t saved_bytes, const float* dy, float* dx, float* grads,
                              int32_t accumulate, double* grad_sq, void* ws, size_t ws_bytes,
                              void* stream) {
  std::string why;
  if (!cfg_ok(cfg, &why)) return fail(RDT_EINVAL, "config: %s", why.c_str());
  if (batch < 1 || seq < 1) return fail(RDT_EINVAL, "batch and seq must be >= 1");
  if (!w || !w_bf16 || !x || !saved || !dy || !dx || !grads || !ws)
    return fail(RDT_EINVAL, "null pointer");
  if (!aligned16(w) || !aligned16(w_bf16) || !aligned16(x) || !aligned16(dy) || !aligned16(dx) ||
      !aligned16(grads) || (reinterpret_cast<uintptr_t>(saved) & 255) ||
      (reinterpret_cast<uintptr_t>(ws) & 255))
    return fail(RDT_EINVAL, "pointers must be 16-byte (saved/ws 256-byte) aligned");
  const Dims m = dims_of(cfg);
  if (saved_bytes < carve_saved(m, batch, seq, nullptr, nullptr))
    return fail(RDT_EINVAL, "saved buffer too small");
  if (ws_bytes < carve_block_ws(m, batch, seq, nullptr, nullptr))
    return fail(RDT_EINVAL, "workspace too small");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = device_error_ptr();
  const int T = batch * seq;
  Saved sv;
  carve_saved(m, batch, seq, const_cast<void*>(saved), &sv);
  BlockWs wk;
  carve_block_ws(m, batch, seq, ws, &wk);
  int64_t off[RDT_BLOCK_NTENSORS];
  block_offsets(m, off);
  const bf16* wb = reinterpret_cast<const bf16*>(w_bf16);

  // dy as a bf16 GEMM operand
  RDT_CHECK_CUDA(cast_bf16(dy, wk.dy_b, (int64_t)T * m.H, s));
  // ds = dy Wd, with the SwiGLU backward in the epilogue -> dgu = [dg | du]
  {
    Epi e;
    e.kind = EPI_SWIGLU_BWD;
    e.out = wk.dgu;
    e.ld_out = 2 * m.I;
    e.aux = sv.gu;
    e.ld_aux = 2 * m.I;
    e.half = (int)m.I;
    RDT_GEMM(Mat{wk.dy_b, T, m.H, m.H}, false, Mat{wb + off[RDT_WD], m.H, m.I, m.I}, true, T,
             (int)m.I, (int)m.H, e, err, s);
  }
  // squared sums of the weight gradients, written by their GEMMs' epilogues
  int64_t sq_n = 0, sq_cnt = 0;
  // a weight gradient: fp32 (+= the previous micro-batches' when accumulating)
  // with its squared-sum slots
  auto sq_slots = [&](Epi& e) {
    if (accumulate) {
      e.kind = EPI_F32_RESID;
      e.resid = static_cast<const float*>(e.out);
      e.ld_resid = e.ld_out;
    }
    if (!grad_sq) return;
    e.sq_part = wk.sqp + sq_n;
    e.sq_count = &sq_cnt;
  };
  // dWd = dy^T s
  {
    Epi e;
    e.kind = EPI_F32;
    e.out = grads + off[RDT_WD];
    e.ld_out = m.I;
    sq_slots(e);
    RDT_GEMM(Mat{wk.dy_b, T, m.H, m.H}, true, Mat{sv.s, T, m.I, m.I}, true, (int)m.H, (int)m.I, T,
             e, err, s);
    if (grad_sq) sq_n += sq_cnt;
  }
  // dxn2 = [dg du] [Wg; Wu]
  {
    Epi e;
    e.kind = EPI_F32;
    e.out = wk.dxn;
    e.ld_out = m.H;
    e.split_ws = wk.split;
    e.split_ws_floats = wk.split_floats;
    RDT_GEMM(Mat{wk.dgu, T, 2 * m.I, 2 * m.I}, false, Mat{wb + off[RDT_WG], 2 * m.I, m.H, m.H},
             true, T, (int)m.H, (int)(2 * m.I), e, err, s);
  }
  // [dWg; dWu] = [dg du]^T xn2
  {
    Epi e;
    e.kind = EPI_F32;
    e.out = grads + off[RDT_WG];
    e.ld_out = m.H;
    sq_slots(e);
    RDT_GEMM(Mat{wk.dgu, T, 2 * m.I, 2 * m.I}, true, Mat{sv.xn2, T, m.H, m.H}, true,
             (int)(2 * m.I), (int)m.H, T, e, err, s);
    if (grad_sq) sq_n += sq_cnt;
  }
  // post-attention RMSNorm backward, identity skip added after it
  RDT_CHECK_CUDA(rmsnorm_bwd(wk.dxn, sv.r1, sv.rstd2, w + off[RDT_G_FFN], dy, wk.dr1, wk.dr1_b,
                             grads + off[RDT_G_FFN], wk.partials, T, (int)m.H, s, accumulate != 0));
  // do = dr1 Wo
  {
    Epi e;
    e.kind = EPI_BF16;
    e.out = wk.dout;
    e.ld_out = m.qd;
    RDT_GEMM(Mat{wk.dr1_b, T, m.H, m.H}, false, Mat{wb + off[RDT_WO], m.H, m.qd, m.qd}, true, T,
             (int)m.qd, (int)m.H, e, err, s);
  }
  // dWo = dr1^T o
  {
    Epi e;
    e.kind = EPI_F32;
    e.out = grads + off[RDT_WO];
    e.ld_out = m.qd;
    sq_slots(e);
    RDT_GEMM(Mat{wk.dr1_b, T, m.H, m.H}, true, Mat{sv.o, T, m.qd, m.qd}, true, (int)m.H,
             (int)m.qd, T, e, err, s);
    if (grad_sq) sq_n += sq_cnt;
  }
  // attention backward (GQA reduction inside), dq accumulated in fp32
  if (attn_tc_supported((int)m.d, true)) {
    // tensor-core backward: padded log2-LSE / D rows (the pre-pass writes the
    // padding as 0); every dq element written once
    const int S_pad = attn_lse_pad(seq);
    RDT_CHECK_CUDA(attn_bwd_pre(sv.o, wk.dout, sv.lse, wk.Dd, wk.lse2, batch, seq, S_pad,
                                (int)m.nh, (int)m.d, s));
    RDT_CHECK_CUDA(attn_bwd_tc(sv.qr, m.qd, sv.kr, m.kd, sv.vb, m.kd, wk.dout,
                               wk.lse2, wk.Dd, wk.dq, wk.dk, wk.dqkv + m.qd + m.kd, m.nqkv, batch,
                               seq, (int)m.nh, (int)m.nkv, (int)m.d, err, s));
  } else {
    RDT_CHECK_CUDA(attn_bwd_pre(sv.o, wk.dout, sv.lse, wk.Dd, nullptr, batch, seq, seq,
                                (int)m.nh, (int)m.d, s));
    RDT_CHECK_CUDA(cudaMemsetAsync(wk.dq, 0, sizeof(float) * T * m.qd, s));
    RDT_CHECK_CUDA(attn_bwd(sv.qr, m.qd, sv.kr, m.kd, sv.vb, m.kd, wk.dout,
                            sv.lse, wk.Dd, wk.dq, wk.dk, wk.dqkv + m.qd + m.kd, m.nqkv, batch, seq,
                            (int)m.nh, (int)m.nkv, (int)m.d, s));
  }
  // inverse RoPE + QK-norm backward -> dq, dk columns of dqkv; q/k gain grads
  RDT_CHECK_CUDA(rope_table(wk.cs, seq, (int)m.d, cfg->rope_theta, s));
  RDT_CHECK_CUDA(qknorm_rope_bwd(wk.dq, wk.dk, sv.qkv, m.nqkv, sv.rstd_q, sv.rstd_k,
                                 w + off[RDT_G_Q], w + off[RDT_G_K], wk.cs, wk.dqkv,
                                 grads + off[RDT_G_Q], wk.partials, T, seq, (int)m.nh, (int)m.nkv,
                                 (int)m.d, s, accumulate != 0));
  // dxn = [dq dk dv] [Wq; Wk; Wv]
  {
    Epi e;
    e.kind = EPI_F32;
    e.out = wk.dxn;
    e.ld_out = m.H;
    e.split_ws = wk.split;
    e.split_ws_floats = wk.split_floats;
    RDT_GEMM(Mat{wk.dqkv, T, m.nqkv, m.nqkv}, false, Mat{wb + off[RDT_WQ], m.nqkv, m.H, m.H}, true,
             T, (int)m.H, (int)m.nqkv, e, err, s);
  }
  // [dWq; dWk; dWv] = [dq dk dv]^T xn
  {
    Epi e;
    e.kind = EPI_F32;
    e.out = grads + off[RDT_WQ];
    e.ld_out = m.H;
    sq_slots(e);
    RDT_GEMM(Mat{wk.dqkv, T, m.nqkv, m.nqkv}, true, Mat{sv.xn, T, m.H, m.H}, true, (int)m.nqkv,
             (int)m.H, T, e, err, s);
    if (grad_sq) sq_n += sq_cnt;
  }
  // input RMSNorm backward + identity skip
  RDT_CHECK_CUDA(rmsnorm_bwd(wk.dxn, x, sv.rstd1, w + off[RDT_G_ATTN], wk.dr1, dx, nullptr,
                             grads + off[RDT_G_ATTN], wk.partials, T, (int)m.H, s, accumulate != 0));
  if (grad_sq) {
    // += the weight-gradient slots and the four gains, in a fixed order
    const float* gains[4] = {grads + off[RDT_G_ATTN], grads + off[RDT_G_FFN],
                             grads + off[RDT_G_Q], grads + off[RDT_G_K]};
    const int64_t lens[4] = {m.H, m.H, m.d, m.d};
    RDT_CHECK_CUDA(sq_reduce(wk.sqp, sq_n, gains, lens, 4, grad_sq, true, wk.sq2, s));
  }
  return RDT_OK;
}

// --------------------------------------------------------------- LM head
rdt_status rdt_fused_cross_entropy(const rdt_config* cfg, int32_t tokens, const float* h,
                                   const float* gamma_f, const rdt_bf16* w_lm,
                                   const int32_t* targets, float loss_scale, float* loss_partials,
                                   float* dh, float* dgamma_f, float* dw_lm, int32_t accumulate,
                                   double* grad_sq, void* ws, size_t ws_bytes, void* stream) {
  std::string why;
  if (!cfg_ok(cfg, &why)) return fail(RDT_EINVAL, "config: %s", why.c_str());
  if (tokens < 1) return fail(RDT_EINVAL, "tokens must be >= 1");
  if (!h || !gamma_f || !w_lm || !targets || !loss_partials || !dh || !dgamma_f || !dw_lm || !ws)
    return fail(RDT_EINVAL, "null pointer");
  if (!aligned16(h) || !aligned16(gamma_f) || !aligned16(w_lm) || !aligned16(dh) ||
      !aligned16(dw_lm) || (reinterpret_cast<uintptr_t>(ws) & 255))
    return fail(RDT_EINVAL, "pointers must be 16-byte (ws 256-byte) aligned");
  const Dims m = dims_of(cfg);
  if (ws_bytes < carve_head_ws(m, tokens, nullptr, nullptr))
    return fail(RDT_EINVAL, "workspace too small");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = device_error_ptr();
  const int T = tokens;
  HeadWs wk;
  carve_head_ws(m, T, ws, &wk);
  const bf16* wl = reinterpret_cast<const bf16*>(w_lm);

  RDT_CHECK_CUDA(rmsnorm_fwd(h, gamma_f, wk.hn, wk.rstd, T, (int)m.H, cfg->rms_eps, s));
  // The logits z = hn W_lm^T are never stored: each GEMM below recomputes a
  // vocabulary chunk of them in its tensor-memory accumulator and its
  // epilogue keeps only what the loss or the gradient needs.
  // Forward: per-row log-sum-exp over the chunks, and the target's logit.
  for (int64_t v0 = 0; v0 < m.V; v0 += wk.vc) {
    const int nv = (int)std::min(wk.vc, m.V - v0);
    Epi e;
    e.kind = EPI_CE;
    e.part = wk.part;
    e.part_ld = wk.part_ld;
    e.targets = targets;
    e.tgt_logit = wk.tgt;
    e.col_off = (int)v0;
    RDT_GEMM(Mat{wk.hn, T, m.H, m.H}, false, Mat{wl + v0 * m.H, nv, m.H, m.H}, false, T, nv,
             (int)m.H, e, err, s);
    RDT_CHECK_CUDA(ce_merge(wk.part, wk.part_ld, ce_partials_per_row(nv), wk.run, v0 == 0,
                            v0 + nv >= m.V, wk.tgt, wk.lse, loss_partials, T, s));
  }
  // Backward, chunk by chunk: dz = loss_scale (softmax(z) - onehot(target))
  // from the recomputed fp32 logits, then dhn += dz W_lm[chunk] and
  // dW_lm[chunk] = dz^T hn.
  int64_t sq_n = 0;
  for (int64_t v0 = 0; v0 < m.V; v0 += wk.vc) {
    const int nv = (int)std::min(wk.vc, m.V - v0);
    const bf16* wc = wl + v0 * m.H;
    {
      Epi e;
      e.kind = EPI_CE_GRAD;
      e.out = wk.dz;
      e.ld_out = wk.vc;
      e.lse = wk.lse;
      e.targets = targets;
      e.col_off = (int)v0;
      e.scale = loss_scale;
      RDT_GEMM(Mat{wk.hn, T, m.H, m.H}, false, Mat{wc, nv, m.H, m.H}, false, T, nv, (int)m.H, e,
               err, s);
    }
    {
      Epi e;
      e.kind = v0 == 0 ? EPI_F32 : EPI_F32_RESID;
      e.out = wk.dhn;
      e.ld_out = m.H;
      e.resid = wk.dhn;
      e.ld_resid = m.H;
      e.split_ws = wk.split;
      e.split_ws_floats = wk.split_floats;
      RDT_GEMM(Mat{wk.dz, T, nv, wk.vc}, false, Mat{wc, nv, m.H, m.H}, true, T, (int)m.H, nv, e,
               err, s);
    }
    {
      Epi e;
      e.kind = accumulate ? EPI_F32_RESID : EPI_F32;
      e.out = dw_lm + v0 * m.H;
      e.ld_out = m.H;
      e.resid = dw_lm + v0 * m.H;
      e.ld_resid = m.H;
      int64_t cnt = 0;
      if (grad_sq) {
        e.sq_part = wk.sqp + sq_n;
        e.sq_count = &cnt;
      }
      RDT_GEMM(Mat{wk.dz, T, nv, wk.vc}, true, Mat{wk.hn, T, m.H, m.H}, true, nv, (int)m.H, T, e,
               err, s);
      sq_n += cnt;
    }
  }
  RDT_CHECK_CUDA(rmsnorm_bwd(wk.dhn, h, wk.rstd, gamma_f, nullptr, dh, nullptr, dgamma_f,
                             wk.partials, T, (int)m.H, s, accumulate != 0));
  if (grad_sq) {
    // = the dW_lm slots and the final gain's squares (the first gradients of a step)
    const float* gains[1] = {dgamma_f};
    const int64_t lens[1] = {m.H};
    RDT_CHECK_CUDA(sq_reduce(wk.sqp, sq_n, gains, lens, 1, grad_sq, false, wk.sq2, s));
  }
  return RDT_OK;
}

// ------------------------------------------------------------ clip / AdamW
rdt_status rdt_sq_sum(const float* const* bufs, const int64_t* lens, int32_t nbuf, double* sumsq,
                      void* ws, size_t ws_bytes, void* stream) {
  if (!bufs || !lens || !sumsq || !ws) return fail(RDT_EINVAL, "null pointer");
  if (nbuf < 1 || nbuf > 64) return fail(RDT_EINVAL, "nbuf must be in [1, 64]");
  if (ws_bytes < sizeof(double)) return fail(RDT_EINVAL, "workspace too small");
  for (int i = 0; i < nbuf; ++i) {
    if (lens[i] < 0 || (lens[i] > 0 && !bufs[i])) return fail(RDT_EINVAL, "bad buffer %d", i);
    if (!aligned16(bufs[i])) return fail(RDT_EINVAL, "buffer %d not 16-byte aligned", i);
  }
  if (reinterpret_cast<uintptr_t>(ws) & 7) return fail(RDT_EINVAL, "workspace not 8-byte aligned");
  int maxp = static_cast<int>(ws_bytes / sizeof(double));
  if (maxp > kMaxSqSumPartials) maxp = kMaxSqSumPartials;
  RDT_CHECK_CUDA(sq_sum(bufs, lens, nbuf, sumsq, static_cast<double*>(ws), maxp,
                        static_cast<cudaStream_t>(stream)));
  return RDT_OK;
}

rdt_status rdt_clip_scale(const double* sumsq, float max_norm, float* scale, int32_t* nonfinite,
                          void* stream) {
  if (!sumsq || !scale) return fail(RDT_EINVAL, "null pointer");
  if (!(max_norm > 0.f)) return fail(RDT_EINVAL, "max_norm must be > 0");
  RDT_CHECK_CUDA(clip_scale(sumsq, max_norm, scale, nonfinite, static_cast<cudaStream_t>(stream)));
  return RDT_OK;
}

rdt_status rdt_adamw_step(float* w, const float* g, float* m, float* v, int64_t n,
                          const float* scale, const int32_t* skip_flag, int32_t step,
                          const int32_t* step_dev, float lr, float beta1, float beta2, float eps,
                          float weight_decay, rdt_bf16* w_bf16, void* stream) {
  if (!w || !g || !m || !v) return fail(RDT_EINVAL, "null pointer");
  if (n < 0) return fail(RDT_EINVAL, "n must be >= 0");
  if (!step_dev && step < 1) return fail(RDT_EINVAL, "step must be >= 1 (bias correction)");
  if (step < 1) step = 1;  // ignored: the kernel reads *step_dev
  if (!aligned16(w) || !aligned16(g) || !aligned16(m) || !aligned16(v) ||
      (w_bf16 && !aligned16(w_bf16)))
    return fail(RDT_EINVAL, "buffers must be 16-byte aligned");
  if (n == 0) return RDT_OK;
  const double bc1 = 1.0 - std::pow(static_cast<double>(beta1), step);
  const double bc2 = 1.0 - std::pow(static_cast<double>(beta2), step);
  RDT_CHECK_CUDA(adamw(w, g, m, v, n, scale, skip_flag, lr, beta1, beta2, eps, weight_decay,
                       static_cast<float>(bc1), static_cast<float>(bc2),
                       reinterpret_cast<bf16*>(w_bf16), static_cast<cudaStream_t>(stream),
                       step_dev));
  return RDT_OK;
}

rdt_status rdt_step_advance(int32_t* step, void* stream) {
  if (!step) return fail(RDT_EINVAL, "null pointer");
  RDT_CHECK_CUDA(step_advance(step, static_cast<cudaStream_t>(stream)));
  return RDT_OK;
}

rdt_status rdt_gemm(const rdt_bf16* A, int32_t a_mn, int64_t lda, const rdt_bf16* B,
                    int32_t b_mn, int64_t ldb, int32_t M, int32_t N, int32_t K, float* C,
                    int64_t ldc, float* split_ws, int64_t split_ws_floats, void* stream) {
  if (!A || !B || !C) return fail(RDT_EINVAL, "null pointer");
  if (M < 1 || N < 1 || K < 1) return fail(RDT_EINVAL, "M, N, K must be >= 1");
  if (lda % 8 || ldb % 8 || ldc % 4 || !aligned16(A) || !aligned16(B) || !aligned16(C))
    return fail(RDT_EINVAL, "lda/ldb must be multiples of 8, ldc of 4, pointers 16-byte aligned");
  const int64_t arows = a_mn ? K : M, acols = a_mn ? M : K;
  const int64_t brows = b_mn ? K : N, bcols = b_mn ? N : K;
  if (lda < acols || ldb < bcols || ldc < N) return fail(RDT_EINVAL, "leading dimension too small");
  if (split_ws && (!aligned16(split_ws) || split_ws_floats < 0))
    return fail(RDT_EINVAL, "split_ws must be 16-byte aligned with a non-negative size");
  Epi e;
  e.kind = EPI_F32;
  e.out = C;
  e.ld_out = ldc;
  e.split_ws = split_ws;
  e.split_ws_floats = split_ws ? split_ws_floats : 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = device_error_ptr();
  RDT_GEMM(Mat{A, arows, acols, lda}, a_mn != 0, Mat{B, brows, bcols, ldb}, b_mn != 0, M, N, K, e,
           err, s);
  return RDT_OK;
}

rdt_status rdt_gemm_nf4(const rdt_bf16* A, int64_t lda, const uint8_t* codes,
                        const float* scales, int64_t w_rows, int64_t w_cols, int32_t b_mn,
                        const rdt_bf16* A2, int64_t lda2, const rdt_bf16* B2, int64_t ldb2,
                        int32_t K2, int32_t M, float* C, int64_t ldc, float* split_ws,
                        int64_t split_ws_floats, void* stream) {
  if (!A || !codes || !scales || !C) return fail(RDT_EINVAL, "null pointer");
  if (M < 1 || w_rows < 1 || w_cols < 1) return fail(RDT_EINVAL, "M and W's dims must be >= 1");
  if (K2 < 0 || K2 > 64 || (K2 > 0 && (!A2 || !B2)))
    return fail(RDT_EINVAL, "K2 must be in [0, 64] with A2 and B2 given when K2 > 0");
  if (w_cols % 256 || w_rows % 64) return fail(RDT_EINVAL, "W needs cols % 256 == 0, rows % 64 == 0");
  const int64_t N = b_mn ? w_cols : w_rows, K1 = b_mn ? w_rows : w_cols;
  if (lda % 8 || ldc % 4 || lda < K1 || ldc < N || !aligned16(A) || !aligned16(C) ||
      !aligned16(codes) || !aligned16(scales))
    return fail(RDT_EINVAL, "lda >= K (multiple of 8), ldc >= N (multiple of 4), 16-byte pointers");
  if (K2 > 0 && (lda2 % 8 || ldb2 % 8 || lda2 < K2 || ldb2 < (b_mn ? N : K2) ||
                 !aligned16(A2) || !aligned16(B2)))
    return fail(RDT_EINVAL, "tail operands: lda2 >= K2, ldb2 >= its row length, multiples of 8");
  if (split_ws && (!aligned16(split_ws) || split_ws_floats < 0))
    return fail(RDT_EINVAL, "split_ws must be 16-byte aligned with a non-negative size");
  Epi e;
  e.kind = EPI_F32;
  e.out = C;
  e.ld_out = ldc;
  e.split_ws = split_ws;
  e.split_ws_floats = split_ws ? split_ws_floats : 0;
  const Mat a{A, M, K1, lda};
  const Mat a2{A2, M, K2, lda2};
  const Mat b2{B2, b_mn ? K2 : N, b_mn ? N : K2, ldb2};
  const char* why = "";
  const cudaError_t ce = gemm_nf4(a, Nf4Mat{codes, scales, w_rows, w_cols}, b_mn != 0,
                                  K2 > 0 ? &a2 : nullptr, K2 > 0 ? &b2 : nullptr, K2, M, e,
                                  device_error_ptr(), static_cast<cudaStream_t>(stream), &why);
  if (ce == cudaErrorInvalidValue && why[0]) return fail(RDT_EINVAL, "%s", why);
  if (ce != cudaSuccess) return fail(RDT_ECUDA, "%s", cudaGetErrorString(ce));
  return RDT_OK;
}

// ---------------------------------------------------------------- embedding
size_t rdt_embedding_workspace_bytes(int32_t tokens) {
  return tokens < 1 ? 0 : embedding_workspace_bytes(tokens);
}

rdt_status rdt_embedding_forward(const float* table, int64_t vocab, int32_t hidden,
                                 const int32_t* ids, int32_t tokens, float* x, void* stream) {
  if (!table || !ids || !x) return fail(RDT_EINVAL, "null pointer");
  if (vocab < 1 || hidden < 4 || hidden % 4 || tokens < 1)
    return fail(RDT_EINVAL, "vocab >= 1, hidden a positive multiple of 4, tokens >= 1");
  if (!aligned16(table) || !aligned16(x)) return fail(RDT_EINVAL, "table and x must be 16-byte aligned");
  RDT_CHECK_CUDA(embedding_forward(table, vocab, hidden, ids, tokens, x, device_error_ptr(),
                                   static_cast<cudaStream_t>(stream)));
  return RDT_OK;
}

rdt_status rdt_embedding_backward(const int32_t* ids, int32_t tokens, const float* dx,
                                  int32_t hidden, const float* scale, float* dtable,
                                  int64_t vocab, int32_t accumulate, void* ws, size_t ws_bytes,
                                  void* stream) {
  if (!ids || !dx || !dtable || !ws) return fail(RDT_EINVAL, "null pointer");
  if (vocab < 1 || hidden < 4 || hidden % 4 || tokens < 1)
    return fail(RDT_EINVAL, "vocab >= 1, hidden a positive multiple of 4, tokens >= 1");
  if (!aligned16(dx) || !aligned16(dtable) || (reinterpret_cast<uintptr_t>(ws) & 255))
    return fail(RDT_EINVAL, "dx, dtable 16-byte and ws 256-byte aligned");
  if (ws_bytes < embedding_workspace_bytes(tokens)) return fail(RDT_EINVAL, "workspace too small");
  RDT_CHECK_CUDA(embedding_backward(ids, tokens, dx, hidden, scale, dtable, vocab,
                                    accumulate != 0, ws, static_cast<cudaStream_t>(stream)));
  return RDT_OK;
}

rdt_status rdt_cast_bf16(const float* src, rdt_bf16* dst, int64_t n, void* stream) {
  if (!src || !dst) return fail(RDT_EINVAL, "null pointer");
  if (n < 0) return fail(RDT_EINVAL, "n must be >= 0");
  if (!aligned16(src) || !aligned16(dst)) return fail(RDT_EINVAL, "buffers must be 16-byte aligned");
  if (n == 0) return RDT_OK;
  RDT_CHECK_CUDA(cast_bf16(src, reinterpret_cast<bf16*>(dst), n, static_cast<cudaStream_t>(stream)));
  return RDT_OK;
}

rdt_status rdt_wait_probe(int64_t limit_ns, int32_t arrive, uint64_t* waited_ns, void* stream) {
  if (limit_ns < 1000 || limit_ns > 10000000000LL)
    return fail(RDT_EINVAL, "limit_ns must be in [1 us, 10 s]");
  if (waited_ns && (reinterpret_cast<uintptr_t>(waited_ns) & 7))
    return fail(RDT_EINVAL, "waited_ns must be 8-byte aligned");
  int* err = device_error_ptr();
  if (!err) return fail(RDT_ECUDA, "device error word not available");
  RDT_CHECK_CUDA(wait_probe(err, static_cast<uint64_t>(limit_ns), arrive != 0,
                            reinterpret_cast<unsigned long long*>(waited_ns),
                            static_cast<cudaStream_t>(stream)));
  return RDT_OK;
}

rdt_status rdt_device_error(int32_t* code) {
  if (!code) return fail(RDT_EINVAL, "null pointer");
  RDT_CHECK_CUDA(cudaDeviceSynchronize());
  int v = 0;
  RDT_CHECK_CUDA(cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)));
  const int zero = 0;
  RDT_CHECK_CUDA(cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)));
  *code = v;
  return RDT_OK;
}

// ------------------------------------------------- NF4 + LoRA block: layout
rdt_status rdt_nf4_check(const rdt_config* cfg, int32_t rank) {
  std::string why;
  if (!nf4_ok(cfg, rank, &why)) return fail(RDT_EINVAL, "%s", why.c_str());
  return RDT_OK;
}

int64_t rdt_nf4_code_bytes(const rdt_config* cfg) {
  std::string why;
  if (!nf4_ok(cfg, 16, &why)) return -1;
  int64_t c;
  nf4_layout(dims_of(cfg), nullptr, nullptr, &c, nullptr);
  return c;
}

int64_t rdt_nf4_scale_count(const rdt_config* cfg) {
  std::string why;
  if (!nf4_ok(cfg, 16, &why)) return -1;
  int64_t sc;
  nf4_layout(dims_of(cfg), nullptr, nullptr, nullptr, &sc);
  return sc;
}

rdt_status rdt_nf4_offsets(const rdt_config* cfg, int64_t* code_offsets, int64_t* scale_offsets) {
  std::string why;
  if (!nf4_ok(cfg, 16, &why)) return fail(RDT_EINVAL, "%s", why.c_str());
  if (!code_offsets || !scale_offsets) return fail(RDT_EINVAL, "null pointer");
  nf4_layout(dims_of(cfg), code_offsets, scale_offsets, nullptr, nullptr);
  return RDT_OK;
}

int64_t rdt_lora_param_count(const rdt_config* cfg, int32_t rank) {
  std::string why;
  if (!nf4_ok(cfg, rank, &why)) return -1;
  int64_t off[RDT_LORA_NTENSORS], cnt[RDT_LORA_NTENSORS];
  lora_layout(dims_of(cfg), rank, off, cnt);
  return off[RDT_LORA_NTENSORS - 1] + cnt[RDT_LORA_NTENSORS - 1];
}

rdt_status rdt_lora_param_offsets(const rdt_config* cfg, int32_t rank, int64_t* offsets,
                                  int64_t* counts) {
  std::string why;
  if (!nf4_ok(cfg, rank, &why)) return fail(RDT_EINVAL, "%s", why.c_str());
  if (!offsets || !counts) return fail(RDT_EINVAL, "null pointer");
  lora_layout(dims_of(cfg), rank, offsets, counts);
  return RDT_OK;
}

int64_t rdt_lora_shadow_count(const rdt_config* cfg, int32_t rank) {
  std::string why;
  if (!nf4_ok(cfg, rank, &why)) return -1;
  return lora_shadow_layout(dims_of(cfg), rank, nullptr).total;
}

rdt_status rdt_lora_shadow(const rdt_config* cfg, int32_t rank, const float* lora,
                           rdt_bf16* shadow, void* stream) {
  std::string why;
  if (!nf4_ok(cfg, rank, &why)) return fail(RDT_EINVAL, "%s", why.c_str());
  if (!lora || !shadow) return fail(RDT_EINVAL, "null pointer");
  if (!aligned16(lora) || !aligned16(shadow)) return fail(RDT_EINVAL, "pointers must be 16-byte aligned");
  const Dims m = dims_of(cfg);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bf16* base = reinterpret_cast<bf16*>(shadow);
  const LoraShadow L = lora_shadow_layout(m, rank, base);
  int64_t off[RDT_LORA_NTENSORS], cnt[RDT_LORA_NTENSORS];
  lora_layout(m, rank, off, cnt);
  // the A's keep their layout; the B's become the stacked tail operands
  RDT_CHECK_CUDA(cast_bf16(lora, base, off[RDT_LORA_B_Q], s));
  {
    const float* p[3] = {lora + off[RDT_LORA_B_Q], lora + off[RDT_LORA_B_K], lora + off[RDT_LORA_B_V]};
    const int64_t rows[3] = {m.qd, m.kd, m.kd};
    RDT_CHECK_CUDA(lora_bstack(p, rows, 3, rank, const_cast<bf16*>(L.b_qkv), s));
  }
  RDT_CHECK_CUDA(cast_bf16(lora + off[RDT_LORA_B_O], const_cast<bf16*>(L.b_o), m.H * rank, s));
  {
    const float* p[2] = {lora + off[RDT_LORA_B_G], lora + off[RDT_LORA_B_U]};
    const int64_t rows[2] = {m.I, m.I};
    RDT_CHECK_CUDA(lora_bstack(p, rows, 2, rank, const_cast<bf16*>(L.b_gu), s));
  }
  RDT_CHECK_CUDA(cast_bf16(lora + off[RDT_LORA_B_D], const_cast<bf16*>(L.b_d), m.H * rank, s));
  return RDT_OK;
}

size_t rdt_nf4_saved_bytes(const rdt_config* cfg, int32_t rank, int32_t batch, int32_t seq) {
  std::string why;
  if (!nf4_ok(cfg, rank, &why) || batch < 1 || seq < 1) return 0;
  return carve_nf4_saved(dims_of(cfg), rank, batch, seq, nullptr, nullptr, nullptr);
}

size_t rdt_nf4_workspace_bytes(const rdt_config* cfg, int32_t rank, int32_t batch, int32_t seq) {
  std::string why;
  if (!nf4_ok(cfg, rank, &why) || batch < 1 || seq < 1) return 0;
  return carve_nf4_ws(dims_of(cfg), rank, batch, seq, nullptr, nullptr, nullptr);
}

// ------------------------------------------------ NF4 + LoRA block: forward
rdt_status rdt_nf4_block_forward(const rdt_config* cfg, int32_t rank, float alpha, int32_t batch,
                                 int32_t seq, const uint8_t* codes, const float* scales,
                                 const float* gains, const rdt_bf16* shadow, const float* x,
                                 float* y, void* saved, size_t saved_bytes, void* ws,
                                 size_t ws_bytes, void* stream) {
  std::string why;
  if (!nf4_ok(cfg, rank, &why)) return fail(RDT_EINVAL, "%s", why.c_str());
  if (batch < 1 || seq < 1) return fail(RDT_EINVAL, "batch and seq must be >= 1");
  if (!(alpha == alpha)) return fail(RDT_EINVAL, "alpha must be a number");
  if (!codes || !scales || !gains || !shadow || !x || !y || !saved || !ws)
    return fail(RDT_EINVAL, "null pointer");
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(gains) || !aligned16(shadow) ||
      !aligned16(x) || !aligned16(y) || (reinterpret_cast<uintptr_t>(saved) & 255) ||
      (reinterpret_cast<uintptr_t>(ws) & 255))
    return fail(RDT_EINVAL, "pointers must be 16-byte (saved/ws 256-byte) aligned");
  if (x == y) return fail(RDT_EINVAL, "y must not alias x");
  const Dims m = dims_of(cfg);
  const int64_t r = rank;
  if (saved_bytes < carve_nf4_saved(m, r, batch, seq, nullptr, nullptr, nullptr))
    return fail(RDT_EINVAL, "saved buffer too small");
  if (ws_bytes < carve_nf4_ws(m, r, batch, seq, nullptr, nullptr, nullptr))
    return fail(RDT_EINVAL, "workspace too small");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = device_error_ptr();
  const int T = batch * seq;
  const float sc = alpha / static_cast<float>(rank);
  Saved sv;
  Nf4Saved nv;
  carve_nf4_saved(m, r, batch, seq, saved, &sv, &nv);
  BlockWs wk;
  Nf4Ws nw;
  carve_nf4_ws(m, r, batch, seq, ws, &wk, &nw);
  const LoraShadow L = lora_shadow_layout(m, r, reinterpret_cast<const bf16*>(shadow));
  int64_t co[7], so[7];
  nf4_layout(m, co, so, nullptr, nullptr);
  auto W = [&](int k, int64_t rows, int64_t cols) {
    return Nf4Mat{codes + co[k], scales + so[k], rows, cols};
  };
  const float *g_attn = gains, *g_ffn = gains + m.H, *g_q = gains + 2 * m.H,
              *g_k = gains + 2 * m.H + m.d;
  // U = s x A^T, the adapters' scaled down-projection (bf16 [T, n])
  auto down = [&](const bf16* xin, int64_t in, const bf16* a, int64_t n, bf16* u) -> rdt_status {
    Epi e;
    e.kind = EPI_BF16;
    e.out = u;
    e.ld_out = n;
    e.scale = sc;
    e.split_ws = nw.split;
    e.split_ws_floats = nw.split_floats;
    RDT_GEMM(Mat{xin, T, in, in}, false, Mat{a, n, in, in}, false, T, (int)n, (int)in, e, err, s);
    return RDT_OK;
  };
  rdt_status st;

  // input RMSNorm
  RDT_CHECK_CUDA(rmsnorm_fwd(x, g_attn, sv.xn, sv.rstd1, T, (int)m.H, cfg->rms_eps, s));
  // qkv = xn [Wq; Wk; Wv]^T + U_qkv [Bq 0 0; 0 Bk 0; 0 0 Bv]^T
  if ((st = down(sv.xn, m.H, L.a_qkv, 3 * r, nv.u_qkv)) != RDT_OK) return st;
  {
    Epi e;
    e.kind = EPI_F32;
    e.out = sv.qkv;
    e.ld_out = m.nqkv;
    const Mat a2{nv.u_qkv, T, 3 * r, 3 * r}, b2{L.b_qkv, m.nqkv, 3 * r, 3 * r};
    e.split_ws = nw.split;
    e.split_ws_floats = nw.split_floats;
    RDT_GEMM_NF4(Mat{sv.xn, T, m.H, m.H}, W(0, m.nqkv, m.H), false, &a2, &b2, (int)(3 * r), T, e,
                 err, s);
  }
  // per-head QK RMSNorm + RoPE-neox, causal GQA attention
  RDT_CHECK_CUDA(rope_table(wk.cs, seq, (int)m.d, cfg->rope_theta, s));
  RDT_CHECK_CUDA(qknorm_rope_fwd(sv.qkv, m.nqkv, sv.qr, sv.kr, sv.vb, sv.rstd_q, sv.rstd_k, g_q,
                                 g_k, wk.cs, T, seq, (int)m.nh, (int)m.nkv, (int)m.d,
                                 cfg->rms_eps, s));
  if (attn_tc_supported((int)m.d, false))
    RDT_CHECK_CUDA(attn_fwd_tc(sv.qr, m.qd, sv.kr, m.kd, sv.vb, m.kd, sv.o, sv.lse, batch, seq,
                               (int)m.nh, (int)m.nkv, (int)m.d, err, s));
  else
    RDT_CHECK_CUDA(attn_fwd(sv.qr, m.qd, sv.kr, m.kd, sv.vb, m.kd, sv.o, sv.lse, batch, seq,
                            (int)m.nh, (int)m.nkv, (int)m.d, s));
  // r1 = x + o Wo^T + U_o Bo^T
  if ((st = down(sv.o, m.qd, L.a_o, r, nv.u_o)) != RDT_OK) return st;
  {
    Epi e;
    e.kind = EPI_F32_RESID;
    e.out = sv.r1;
    e.ld_out = m.H;
    e.resid = x;
    e.ld_resid = m.H;
    const Mat a2{nv.u_o, T, r, r}, b2{L.b_o, m.H, r, r};
    e.split_ws = nw.split;
    e.split_ws_floats = nw.split_floats;
    RDT_GEMM_NF4(Mat{sv.o, T, m.qd, m.qd}, W(3, m.H, m.qd), false, &a2, &b2, (int)r, T, e, err, s);
  }
  // post-attention RMSNorm
  RDT_CHECK_CUDA(rmsnorm_fwd(sv.r1, g_ffn, sv.xn2, sv.rstd2, T, (int)m.H, cfg->rms_eps, s));
  // [g | u] = xn2 [Wg; Wu]^T + U_gu [Bg 0; 0 Bu]^T with the SwiGLU epilogue
  if ((st = down(sv.xn2, m.H, L.a_gu, 2 * r, nv.u_gu)) != RDT_OK) return st;
  {
    Epi e;
    e.kind = EPI_SWIGLU;
    e.out = sv.gu;
    e.ld_out = 2 * m.I;
    e.out2 = sv.s;
    e.ld_out2 = m.I;
    e.half = (int)m.I;
    const Mat a2{nv.u_gu, T, 2 * r, 2 * r}, b2{L.b_gu, 2 * m.I, 2 * r, 2 * r};
    RDT_GEMM_NF4(Mat{sv.xn2, T, m.H, m.H}, W(4, 2 * m.I, m.H), false, &a2, &b2, (int)(2 * r), T, e,
                 err, s);
  }
  // y = r1 + s Wd^T + U_d Bd^T
  if ((st = down(sv.s, m.I, L.a_d, r, nv.u_d)) != RDT_OK) return st;
  {
    Epi e;
    e.kind = EPI_F32_RESID;
    e.out = y;
    e.ld_out = m.H;
    e.resid = sv.r1;
    e.ld_resid = m.H;
    const Mat a2{nv.u_d, T, r, r}, b2{L.b_d, m.H, r, r};
    e.split_ws = nw.split;
    e.split_ws_floats = nw.split_floats;
    RDT_GEMM_NF4(Mat{sv.s, T, m.I, m.I}, W(6, m.H, m.I), false, &a2, &b2, (int)r, T, e, err, s);
  }
  return RDT_OK;
}

// ----------------------------------------------- NF4 + LoRA block: backward
rdt_status rdt_nf4_block_backward(const rdt_config* cfg, int32_t rank, float alpha,
                                  int32_t batch, int32_t seq, const uint8_t* codes,
                                  const float* scales, const float* gains,
                                  const rdt_bf16* shadow, const float* x, const void* saved,
                                  size_t saved_bytes, const float* dy, float* dx,
                                  float* lora_grads, double* grad_sq, void* ws, size_t ws_bytes,
                                  void* stream) {
  std::string why;
  if (!nf4_ok(cfg, rank, &why)) return fail(RDT_EINVAL, "%s", why.c_str());
  if (batch < 1 || seq < 1) return fail(RDT_EINVAL, "batch and seq must be >= 1");
  if (!(alpha == alpha)) return fail(RDT_EINVAL, "alpha must be a number");
  if (!codes || !scales || !gains || !shadow || !x || !saved || !dy || !dx || !lora_grads || !ws)
    return fail(RDT_EINVAL, "null pointer");
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(gains) || !aligned16(shadow) ||
      !aligned16(x) || !aligned16(dy) || !aligned16(dx) || !aligned16(lora_grads) ||
      (reinterpret_cast<uintptr_t>(saved) & 255) || (reinterpret_cast<uintptr_t>(ws) & 255))
    return fail(RDT_EINVAL, "pointers must be 16-byte (saved/ws 256-byte) aligned");
  const Dims m = dims_of(cfg);
  const int64_t r = rank;
  if (saved_bytes < carve_nf4_saved(m, r, batch, seq, nullptr, nullptr, nullptr))
    return fail(RDT_EINVAL, "saved buffer too small");
  if (ws_bytes < carve_nf4_ws(m, r, batch, seq, nullptr, nullptr, nullptr))
    return fail(RDT_EINVAL, "workspace too small");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = device_error_ptr();
  const int T = batch * seq;
  const float sc = alpha / static_cast<float>(rank);
  Saved sv;
  Nf4Saved nv;
  carve_nf4_saved(m, r, batch, seq, const_cast<void*>(saved), &sv, &nv);
  BlockWs wk;
  Nf4Ws nw;
  carve_nf4_ws(m, r, batch, seq, ws, &wk, &nw);
  const LoraShadow L = lora_shadow_layout(m, r, reinterpret_cast<const bf16*>(shadow));
  int64_t co[7], so[7];
  nf4_layout(m, co, so, nullptr, nullptr);
  auto W = [&](int k, int64_t rows, int64_t cols) {
    return Nf4Mat{codes + co[k], scales + so[k], rows, cols};
  };
  int64_t lo[RDT_LORA_NTENSORS], lc[RDT_LORA_NTENSORS];
  lora_layout(m, r, lo, lc);
  float* G = lora_grads;
  const float *g_attn = gains, *g_ffn = gains + m.H, *g_q = gains + 2 * m.H,
              *g_k = gains + 2 * m.H + m.d;
  int64_t sq_n = 0, sq_cnt = 0;
  // dU = s dY B (bf16 [T, n]): B as stored, [K = out, N = n]
  auto up = [&](const bf16* dyb, int64_t out, const bf16* b, int64_t n, bf16* du) -> rdt_status {
    Epi e;
    e.kind = EPI_BF16;
    e.out = du;
    e.ld_out = n;
    e.scale = sc;
    e.split_ws = nw.split;
    e.split_ws_floats = nw.split_floats;
    RDT_GEMM(Mat{dyb, T, out, out}, false, Mat{b, out, n, n}, true, T, (int)n, (int)out, e, err,
             s);
    return RDT_OK;
  };
  // C[M, N] = P^T Q over the T tokens (P [T, M], Q [T, N] as stored), fp32 into
  // the adapter gradient at lora_grads + off, with squared-sum slots
  auto tn = [&](const bf16* P, int64_t M, int64_t ldp, const bf16* Q, int64_t N, int64_t ldq,
                int tensor) -> rdt_status {
    Epi e;
    e.kind = EPI_F32;
    e.out = G + lo[tensor];
    e.ld_out = N;
    e.split_ws = nw.split;
    e.split_ws_floats = nw.split_floats;
    if (grad_sq) {
      e.sq_part = nw.sqp + sq_n;
      e.sq_count = &sq_cnt;
    }
    RDT_GEMM(Mat{P, T, M, ldp}, true, Mat{Q, T, N, ldq}, true, (int)M, (int)N, T, e, err, s);
    if (grad_sq) sq_n += sq_cnt;
    return RDT_OK;
  };
  rdt_status st;

  // dy as a bf16 GEMM operand
  RDT_CHECK_CUDA(cast_bf16(dy, wk.dy_b, (int64_t)T * m.H, s));
  // down projection: ds = dy Wd + dU_d Ad with the SwiGLU backward in the epilogue
  if ((st = up(wk.dy_b, m.H, L.b_d, r, nw.du_d)) != RDT_OK) return st;
  {
    Epi e;
    e.kind = EPI_SWIGLU_BWD;
    e.out = wk.dgu;
    e.ld_out = 2 * m.I;
    e.aux = sv.gu;
    e.ld_aux = 2 * m.I;
    e.half = (int)m.I;
    const Mat a2{nw.du_d, T, r, r}, b2{L.a_d, r, m.I, m.I};
    RDT_GEMM_NF4(Mat{wk.dy_b, T, m.H, m.H}, W(6, m.H, m.I), true, &a2, &b2, (int)r, T, e, err, s);
  }
  // dBd = dy^T U_d, dAd = dU_d^T s
  if ((st = tn(wk.dy_b, m.H, m.H, nv.u_d, r, r, RDT_LORA_B_D)) != RDT_OK) return st;
  if ((st = tn(nw.du_d, r, r, sv.s, m.I, m.I, RDT_LORA_A_D)) != RDT_OK) return st;
  // gate/up: dxn2 = [dg du] [Wg; Wu] + dU_gu [Ag; Au]
  if ((st = up(wk.dgu, 2 * m.I, L.b_gu, 2 * r, nw.du_gu)) != RDT_OK) return st;
  {
    Epi e;
    e.kind = EPI_F32;
    e.out = wk.dxn;
    e.ld_out = m.H;
    const Mat a2{nw.du_gu, T, 2 * r, 2 * r}, b2{L.a_gu, 2 * r, m.H, m.H};
    e.split_ws = nw.split;
    e.split_ws_floats = nw.split_floats;
    RDT_GEMM_NF4(Mat{wk.dgu, T, 2 * m.I, 2 * m.I}, W(4, 2 * m.I, m.H), true, &a2, &b2,
                 (int)(2 * r), T, e, err, s);
  }
  // dBg = dg^T U_g, dBu = du^T U_u, [dAg; dAu] = dU_gu^T xn2
  if ((st = tn(wk.dgu, m.I, 2 * m.I, nv.u_gu, r, 2 * r, RDT_LORA_B_G)) != RDT_OK) return st;
  if ((st = tn(wk.dgu + m.I, m.I, 2 * m.I, nv.u_gu + r, r, 2 * r, RDT_LORA_B_U)) != RDT_OK)
    return st;
  if ((st = tn(nw.du_gu, 2 * r, 2 * r, sv.xn2, m.H, m.H, RDT_LORA_A_G)) != RDT_OK) return st;
  // post-attention RMSNorm backward (frozen gain), identity skip added after it
  RDT_CHECK_CUDA(rmsnorm_bwd(wk.dxn, sv.r1, sv.rstd2, g_ffn, dy, wk.dr1, wk.dr1_b, nw.gain_sink,
                             wk.partials, T, (int)m.H, s));
  // O projection: do = dr1 Wo + dU_o Ao (bf16)
  if ((st = up(wk.dr1_b, m.H, L.b_o, r, nw.du_o)) != RDT_OK) return st;
  {
    Epi e;
    e.kind = EPI_BF16;
    e.out = wk.dout;
    e.ld_out = m.qd;
    const Mat a2{nw.du_o, T, r, r}, b2{L.a_o, r, m.qd, m.qd};
    RDT_GEMM_NF4(Mat{wk.dr1_b, T, m.H, m.H}, W(3, m.H, m.qd), true, &a2, &b2, (int)r, T, e, err,
                 s);
  }
  // dBo = dr1^T U_o, dAo = dU_o^T o
  if ((st = tn(wk.dr1_b, m.H, m.H, nv.u_o, r, r, RDT_LORA_B_O)) != RDT_OK) return st;
  if ((st = tn(nw.du_o, r, r, sv.o, m.qd, m.qd, RDT_LORA_A_O)) != RDT_OK) return st;
  // attention backward
  if (attn_tc_supported((int)m.d, true)) {
    const int S_pad = attn_lse_pad(seq);  // the pre-pass writes the padding as 0
    RDT_CHECK_CUDA(attn_bwd_pre(sv.o, wk.dout, sv.lse, wk.Dd, wk.lse2, batch, seq, S_pad,
                                (int)m.nh, (int)m.d, s));
    RDT_CHECK_CUDA(attn_bwd_tc(sv.qr, m.qd, sv.kr, m.kd, sv.vb, m.kd, wk.dout, wk.lse2, wk.Dd,
                               wk.dq, wk.dk, wk.dqkv + m.qd + m.kd, m.nqkv, batch, seq, (int)m.nh,
                               (int)m.nkv, (int)m.d, err, s));
  } else {
    RDT_CHECK_CUDA(attn_bwd_pre(sv.o, wk.dout, sv.lse, wk.Dd, nullptr, batch, seq, seq,
                                (int)m.nh, (int)m.d, s));
    RDT_CHECK_CUDA(cudaMemsetAsync(wk.dq, 0, sizeof(float) * T * m.qd, s));
    RDT_CHECK_CUDA(attn_bwd(sv.qr, m.qd, sv.kr, m.kd, sv.vb, m.kd, wk.dout, sv.lse, wk.Dd, wk.dq,
                            wk.dk, wk.dqkv + m.qd + m.kd, m.nqkv, batch, seq, (int)m.nh,
                            (int)m.nkv, (int)m.d, s));
  }
  // inverse RoPE + QK-norm backward (frozen gains) -> dq, dk columns of dqkv
  RDT_CHECK_CUDA(rope_table(wk.cs, seq, (int)m.d, cfg->rope_theta, s));
  RDT_CHECK_CUDA(qknorm_rope_bwd(wk.dq, wk.dk, sv.qkv, m.nqkv, sv.rstd_q, sv.rstd_k, g_q, g_k,
                                 wk.cs, wk.dqkv, nw.gain_sink + m.H, wk.partials, T, seq,
                                 (int)m.nh, (int)m.nkv, (int)m.d, s));
  // Q/K/V: dxn = dqkv [Wq; Wk; Wv] + dU_qkv [Aq; Ak; Av]
  if ((st = up(wk.dqkv, m.nqkv, L.b_qkv, 3 * r, nw.du_qkv)) != RDT_OK) return st;
  {
    Epi e;
    e.kind = EPI_F32;
    e.out = wk.dxn;
    e.ld_out = m.H;
    const Mat a2{nw.du_qkv, T, 3 * r, 3 * r}, b2{L.a_qkv, 3 * r, m.H, m.H};
    e.split_ws = nw.split;
    e.split_ws_floats = nw.split_floats;
    RDT_GEMM_NF4(Mat{wk.dqkv, T, m.nqkv, m.nqkv}, W(0, m.nqkv, m.H), true, &a2, &b2, (int)(3 * r),
                 T, e, err, s);
  }
  // dBq = dq^T U_q, dBk = dk^T U_k, dBv = dv^T U_v, [dAq; dAk; dAv] = dU_qkv^T xn
  if ((st = tn(wk.dqkv, m.qd, m.nqkv, nv.u_qkv, r, 3 * r, RDT_LORA_B_Q)) != RDT_OK) return st;
  if ((st = tn(wk.dqkv + m.qd, m.kd, m.nqkv, nv.u_qkv + r, r, 3 * r, RDT_LORA_B_K)) != RDT_OK)
    return st;
  if ((st = tn(wk.dqkv + m.qd + m.kd, m.kd, m.nqkv, nv.u_qkv + 2 * r, r, 3 * r, RDT_LORA_B_V)) !=
      RDT_OK)
    return st;
  if ((st = tn(nw.du_qkv, 3 * r, 3 * r, sv.xn, m.H, m.H, RDT_LORA_A_Q)) != RDT_OK) return st;
  // input RMSNorm backward (frozen gain) + identity skip
  RDT_CHECK_CUDA(rmsnorm_bwd(wk.dxn, x, sv.rstd1, g_attn, wk.dr1, dx, nullptr, nw.gain_sink,
                             wk.partials, T, (int)m.H, s));
  if (grad_sq)
    RDT_CHECK_CUDA(sq_reduce(nw.sqp, sq_n, nullptr, nullptr, 0, grad_sq, true, nw.sq2, s));
  return RDT_OK;
}

}  // extern "C"
