// rdt_sq_sum_noalloc: the squared-sum reduction of rdt_sq_sum for callers
// that cannot allocate device memory -- code running where cudaMalloc is not
// allowed or not wanted (inside an allocator or memory-pool callback, a
// runtime that must not grow its footprint once started, a plugin that
// cannot receive a scratch buffer through its host's interface). Its scratch
// (the per-block fp64 partial sums) lives in a fixed array in this file
// instead of a caller workspace.
#include <mutex>

#include "../../include/rdt.h"
#include "internal.h"

namespace {

// Room for the per-block partial sums of one reduction: 4096 fp64 values
// (32 KiB). Every GPU that loads librdt.so keeps this array until the process
// exits. The launch never uses more blocks than this, so any total length is
// accepted; only the 64-buffer table limit can reject a call.
constexpr int kStaticPartials = 4096;
__device__ __align__(256) double g_sq_sum_scratch[kStaticPartials];

// Device address of the array on the current device. In host code the
// symbol is only a host-side stand-in, so the address is looked up once per
// device with that device current and cached.
double* scratch_on_current_device(cudaError_t* err) {
  static double* addr[64] = {};
  static std::mutex mu;
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_sq_sum_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = static_cast<double*>(p);
  }
  return addr[dev];
}

}  // namespace

extern "C" rdt_status rdt_sq_sum_noalloc(const float* const* bufs, const int64_t* lens,
                                         int32_t nbuf, double* sumsq, void* stream) {
  if (!bufs || !lens || !sumsq) {
    rdt::set_last_error("rdt_sq_sum_noalloc: null pointer");
    return RDT_EINVAL;
  }
  if (nbuf < 1 || nbuf > 64) {
    rdt::set_last_error("rdt_sq_sum_noalloc: nbuf must be in [1, 64] (one call sums at most 64 buffers)");
    return RDT_EINVAL;
  }
  for (int i = 0; i < nbuf; ++i) {
    if (lens[i] < 0 || (lens[i] > 0 && !bufs[i]) ||
        (reinterpret_cast<uintptr_t>(bufs[i]) & 15)) {
      rdt::set_last_error("rdt_sq_sum_noalloc: every buffer must be non-null and 16-byte aligned");
      return RDT_EINVAL;
    }
  }
  cudaError_t e = cudaSuccess;
  double* scratch = scratch_on_current_device(&e);
  if (!scratch) {
    rdt::set_last_error(cudaGetErrorString(e));
    return RDT_ECUDA;
  }
  // The reduction writes every partial it later reads, so nothing in the
  // array needs clearing between calls.
  e = rdt::sq_sum(bufs, lens, nbuf, sumsq, scratch, kStaticPartials,
                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    rdt::set_last_error(cudaGetErrorString(e));
    return RDT_ECUDA;
  }
  return RDT_OK;
}
