// Token embedding on the device: lookup (gather) and its backward, a
// deterministic scatter-add of the activation gradient into the table's
// gradient (cuda_trainer.rs: gpu_forward's embedding lookup, embed_backward's
// scatter-add, moved from the host to the GPU).
//
// The backward orders the tokens stably by id (O(T^2) comparisons staged in
// shared memory, no atomics), then one warp per run of equal ids sums that
// run's rows in token order and adds scale x the sum into the id's gradient
// row, so the result does not depend on scheduling.
#include "common.cuh"
#include "internal.h"

namespace rdt {

namespace {

constexpr int kSortTile = 2048;  // ids staged per shared-memory tile

// x[t, :] = table[ids[t], :] (rows of H4 float4). An id outside [0, V)
// gives a zero row and records kErrIndex in the device error word.
__global__ void __launch_bounds__(256) embed_gather_kernel(const float4* __restrict__ table,
                                                          const int32_t* __restrict__ ids,
                                                          int T, int H4, int64_t V,
                                                          float4* __restrict__ x, int* err) {
  const int64_t n = static_cast<int64_t>(T) * H4;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / H4;
    const int64_t c = i - t * H4;
    const int32_t id = ids[t];
    if (id < 0 || id >= V) {
      x[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c == 0) record_error(err, kErrIndex);
    } else {
      x[i] = table[static_cast<int64_t>(id) * H4 + c];
    }
  }
}

// perm[rank(t)] = t with rank(t) = #{t' : (ids[t'], t') < (ids[t], t)}:
// the tokens in stable id order.
__global__ void __launch_bounds__(256) embed_sort_kernel(const int32_t* __restrict__ ids, int T,
                                                        int32_t* __restrict__ perm) {
  __shared__ int32_t tile[kSortTile];
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  const int32_t mine = t < T ? ids[t] : 0;
  int rank = 0;
  for (int base = 0; base < T; base += kSortTile) {
    const int n = min(kSortTile, T - base);
    __syncthreads();
    for (int j = threadIdx.x; j < n; j += blockDim.x) tile[j] = ids[base + j];
    __syncthreads();
    if (t < T) {
      for (int j = 0; j < n; ++j) {
        const int32_t o = tile[j];
        rank += (o < mine) || (o == mine && base + j < t);
      }
    }
  }
  if (t < T) perm[rank] = t;
}

// One warp per position r of the sorted order that starts a run of equal
// ids: dtable[id, :] (= or +=) scale * sum over the run, in token order, of
// dx[t, :]. H % 4 == 0; ids outside [0, V) are skipped.
__global__ void __launch_bounds__(256) embed_scatter_kernel(
    const int32_t* __restrict__ ids, const int32_t* __restrict__ perm, int T,
    const float* __restrict__ dx, int H, const float* __restrict__ scale,
    float* __restrict__ dtable, int64_t V, int accumulate) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const float s = scale ? *scale : 1.0f;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < T; r += warps) {
    const int32_t id = ids[perm[r]];
    if (r > 0 && ids[perm[r - 1]] == id) continue;  // not the start of a run
    if (id < 0 || id >= V) continue;
    int e = r + 1;
    while (e < T && ids[perm[e]] == id) ++e;
    float4* out = reinterpret_cast<float4*>(dtable + static_cast<int64_t>(id) * H);
    for (int c = lane; c < H / 4; c += 32) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int k = r; k < e; ++k) {
        const float4 v =
            reinterpret_cast<const float4*>(dx + static_cast<int64_t>(perm[k]) * H)[c];
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      float4 o = accumulate ? out[c] : make_float4(0.f, 0.f, 0.f, 0.f);
      o.x += s * acc.x;
      o.y += s * acc.y;
      o.z += s * acc.z;
      o.w += s * acc.w;
      out[c] = o;
    }
  }
}

__global__ void __launch_bounds__(256) zero_kernel(float4* __restrict__ p, int64_t n4) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

int grid_for(int64_t items) {
  int64_t b = (items + 255) / 256;
  const int64_t cap = 8LL * num_sms();
  if (b > cap) b = cap;
  return b < 1 ? 1 : static_cast<int>(b);
}

}  // namespace

cudaError_t embedding_forward(const float* table, int64_t V, int H, const int32_t* ids, int T,
                              float* x, int* err, cudaStream_t s) {
  const int H4 = H / 4;
  note_launch();
  embed_gather_kernel<<<grid_for(static_cast<int64_t>(T) * H4), 256, 0, s>>>(
      reinterpret_cast<const float4*>(table), ids, T, H4, V, reinterpret_cast<float4*>(x), err);
  return cudaGetLastError();
}

size_t embedding_workspace_bytes(int T) { return (static_cast<size_t>(T) * 4 + 255) / 256 * 256; }

cudaError_t embedding_backward(const int32_t* ids, int T, const float* dx, int H,
                               const float* scale, float* dtable, int64_t V, bool accumulate,
                               void* ws, cudaStream_t s) {
  int32_t* perm = static_cast<int32_t*>(ws);
  if (!accumulate) {
    // untouched rows of the gradient are zero
    note_launch();
    const int64_t n4 = V * H / 4;
    zero_kernel<<<grid_for(n4), 256, 0, s>>>(reinterpret_cast<float4*>(dtable), n4);
  }
  note_launch();
  embed_sort_kernel<<<(T + 255) / 256, 256, 0, s>>>(ids, T, perm);
  note_launch();
  embed_scatter_kernel<<<grid_for(static_cast<int64_t>(T) * 32), 256, 0, s>>>(
      ids, perm, T, dx, H, scale, dtable, V, 1);
  return cudaGetLastError();
}

}  // namespace rdt
