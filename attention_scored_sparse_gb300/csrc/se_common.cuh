// Shared device/host helpers of the sm_103a kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "se.h"

#define SE_DEV __device__ __forceinline__
#define SE_HD __host__ __device__ __forceinline__

namespace se {

SE_HD int cdiv(int a, int b) { return (a + b - 1) / b; }
SE_HD int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Programmatic dependent launch.  Every kernel is launched with se_launch,
// which lets it start while the kernel before it in the stream is still
// finishing, and every kernel calls pdl_enter before it touches global
// memory: the wait there returns once the previous kernel has completed and
// its writes are visible, and the trigger then lets the next kernel of the
// stream launch early in turn.  The launch latency and the ramp of the next
// grid overlap the tail of the current one; the order of memory accesses is
// that of plain stream order.  (Launched without the attribute, both
// instructions do nothing.)
SE_DEV void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... K, typename... A>
inline cudaError_t se_launch(void (*kernel)(K...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, A&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

// se_launch for a kernel whose CTAs form clusters of `cluster_x` along x
// (the grid's x a multiple of it).
template <typename... K, typename... A>
inline cudaError_t se_launch_cluster(void (*kernel)(K...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t st, int cluster_x, A&&... args) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

// Dynamic shared memory above 48 KB is allowed per kernel and per device:
// sets the limit the first time `kernel` is launched on the current device.
// `done` holds one bit per device (devices past 64 set it on every call).
inline bool allow_smem(const void* kernel, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t{1} << dev) : 0;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return false;
  if (bit != 0) done.fetch_or(bit, std::memory_order_release);
  return true;
}

// First-writer-wins device error word.
SE_DEV void set_status(int32_t* status, int32_t code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

constexpr float kLog2e = 1.4426950408889634f;

// bf16 pair (packed in a uint32) -> two floats, exact.
SE_DEV float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
SE_DEV float bf16hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// 8 consecutive elements (16 bytes for bf16) -> floats.
SE_DEV void unpack8_bf16(const uint4& u, float* f) {
  f[0] = bf16lo(u.x); f[1] = bf16hi(u.x);
  f[2] = bf16lo(u.y); f[3] = bf16hi(u.y);
  f[4] = bf16lo(u.z); f[5] = bf16hi(u.z);
  f[6] = bf16lo(u.w); f[7] = bf16hi(u.w);
}

SE_DEV uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

SE_DEV uint4 ldg_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

SE_DEV void stg_v4(void* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Order-preserving float -> uint32 key (larger float -> larger key).
SE_DEV uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive scan of one int per thread (blockDim.x <= 1024,
// multiple of 32).  `tmp` must hold 33 ints of shared memory.  Returns the
// exclusive prefix; *total receives the block sum.  Contains __syncthreads.
SE_DEV int block_exclusive_scan(int v, int* tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nwarps) tmp[lane] = w;  // inclusive warp totals
    if (lane == 31) tmp[32] = w;
  }
  __syncthreads();
  int base = warp > 0 ? tmp[warp - 1] : 0;
  int t = tmp[32];
  __syncthreads();
  if (total) *total = t;
  return base + x - v;
}

// Counts a thread's keys (ITEMS consecutive candidates) into hist: keys of
// the digit `shift`/`dmask` whose higher digits equal `prefix` (mask
// `pmask`), key 0 = absent.  Runs of one bin are added by one atomic: close
// candidates tend to share a bin, and the lanes of a warp adding to one bin
// at once would serialise.
template <int ITEMS>
SE_DEV void hist_add_keys(int* hist, const uint32_t (&key)[ITEMS], int shift, uint32_t dmask,
                          uint32_t pmask, uint32_t prefix) {
  uint32_t cur = 0xffffffffu;
  int cnt = 0;
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    if (key[i] != 0u && (key[i] & pmask) == prefix) {
      const uint32_t bin = (key[i] >> shift) & dmask;
      if (bin != cur) {
        if (cnt) atomicAdd(&hist[cur], cnt);
        cur = bin;
        cnt = 0;
      }
      ++cnt;
    }
  }
  if (cnt) atomicAdd(&hist[cur], cnt);
}

// Radix-select step: hist[0 .. nbins) holds the candidate count per digit;
// finds the digit that holds the `remaining`-th largest key (counting from
// the top digit down) and how many keys of that digit are still needed.
// Every thread calls it (nbins a multiple of blockDim.x, or below it); one
// block scan replaces a serial walk over the bins.  Results in *s_digit,
// *s_rem (shared), valid after the call.
SE_DEV void radix_find_digit(const int* hist, int nbins, int remaining, int* tmp, int* s_digit,
                             int* s_rem) {
  const int per = nbins >= (int)blockDim.x ? nbins / (int)blockDim.x : 1;
  const int b0 = threadIdx.x * per;
  int c = 0;
  for (int j = 0; j < per; ++j)
    if (b0 + j < nbins) c += hist[b0 + j];
  int total;
  const int ex = block_exclusive_scan(c, tmp, &total);
  const int above = total - ex - c;          // keys in higher digits than this thread's
  if (c > 0 && above < remaining && above + c >= remaining) {
    int acc = above;
    for (int j = per - 1; j >= 0; --j) {
      const int cnt = b0 + j < nbins ? hist[b0 + j] : 0;
      if (acc + cnt >= remaining) {
        *s_digit = b0 + j;
        *s_rem = remaining - acc;
        break;
      }
      acc += cnt;
    }
  }
  __syncthreads();
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bump allocator over a caller-provided workspace (host side).
struct WsCarver {
  char* base;
  size_t off = 0;
  explicit WsCarver(void* p) : base(static_cast<char*>(p)) {}
  template <typename T>
  T* take(size_t n) {
    off = align_up(off, 256);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += n * sizeof(T);
    return p;
  }
  size_t bytes() const { return align_up(off, 256); }
};

SE_HD size_t elem_size(int32_t dtype) { return dtype == SE_BF16 ? 2 : 4; }

}  // namespace se

// Host-side launch helpers shared by the translation units.
se_status se_check_kv(const se_paged_kv* kv);
se_status se_last_launch_status();
