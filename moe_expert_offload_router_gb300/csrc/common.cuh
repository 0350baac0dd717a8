// Shared helpers of the library's translation units (host error handling,
// the cache handle, small device utilities).  Device-side code here performs
// no MoE arithmetic of its own.
#pragma once

#include <utility>

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <stddef.h>

#include "moe_gb300.h"

namespace moe {

constexpr uint32_t kFreqCap = (1u << 20) - 1;  // LFU count cap (20 bits of the eviction order key)


moe_status fail(moe_status s, const char* fmt, ...);
moe_status cuda_fail(cudaError_t e, const char* what);
void clear_error();

// Kernel launch check: a launch error is returned, not printed.
inline moe_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, what);
  return MOE_OK;
}

// Programmatic dependent launch.  A kernel launched with launch_pdl may start
// while the kernel before it on the stream is still running: it must call
// pdl_wait() before it reads or writes anything that kernel touches (the wait
// returns once that kernel has completed and its writes are visible), and a
// kernel calls pdl_launch_dependents() to let the next one start early.  Both
// are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Records a start event now and a stop event when the scope ends, on the
// launching stream, if profiling is enabled (moe_profile_enable).
class ProfScope {
 public:
  ProfScope(int kernel, cudaStream_t s);
  ~ProfScope();

 private:
  int k_;
  cudaStream_t s_;
  void* stop_;
};

size_t fp4_bytes(int H, int I);
size_t int2_bytes(int H, int I);
size_t fp8_bytes(int H, int I);

// Device LRU state of one slot cache, as passed to kernels.
struct CacheDev {
  int32_t* slot_key;     // [S] key held by the slot, -1 = empty
  uint64_t* slot_stamp;  // [S] recency stamp (unique among occupied slots)
  int32_t* key_to_slot;  // [L*E] slot of a key, -1 = not resident
  uint64_t* clock;       // [1]
  uint32_t* freq;        // [L*E] LFU count of a key
  uint32_t* freq_epoch;  // [L*E] epoch in which the count was last written
  uint64_t* calls;       // [1] ensure calls that returned (LFU epochs)
  int S, L, E;
  int policy;            // MOE_EVICT_LRU or MOE_EVICT_LFU
  int decay_calls;       // LFU: counts halve once per this many calls
  int R;                 // staging-ring slots after the S cache slots (0 = none)
  int32_t* stage_key;    // [R] key staged in ring slot j, -1 = none
  int32_t* stage_of;     // [L*E] ring slot holding a key, -1 = not staged
  uint32_t* stage_pos;   // [1] next ring position (mod R)
};

}  // namespace moe

struct moe_cache {
  int S, L, E;
  size_t B;               // bytes per expert
  uint8_t* d_slots;       // caller-owned slot pool
  const uint8_t* h_bank;  // caller-owned pinned bank (may be null)
  void* d_state;          // library-owned block holding the LRU arrays
  moe::CacheDev dev;
  int device;
  int fail_copy_index;    // host-side fault injection for moe_copy_missing (-1 = off)
  const uint8_t* bank_dev;  // device-side address of h_bank (null if not mapped)
  void* d_stage;            // library-owned staging-ring state (null if none)
};

#define MOE_ARG(cond, ...)                                   \
  do {                                                       \
    if (!(cond)) return moe::fail(MOE_ERR_INVALID, __VA_ARGS__); \
  } while (0)

#define MOE_CUDA(call)                                       \
  do {                                                       \
    cudaError_t _e = (call);                                 \
    if (_e != cudaSuccess) return moe::cuda_fail(_e, #call); \
  } while (0)

// ---------------------------------------------------------------------------
// device utilities
// ---------------------------------------------------------------------------
namespace moe {

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  // Streamed weight bytes: read once per launch, keep them out of L1.
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Block-wide exclusive scan of one int per thread (blockDim.x a multiple of 32,
// at most 1024).  `ws` needs 33 ints of shared memory.  Returns the exclusive
// prefix; *total receives the sum.  Contains __syncthreads.
__device__ __forceinline__ int block_exclusive_scan(int v, int* ws, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) ws[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int t = lane < nw ? ws[lane] : 0;
    int ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += n;
    }
    ws[lane] = ti - t;  // exclusive warp offsets
    if (lane == 31) ws[32] = ti;
  }
  __syncthreads();
  int r = ws[wid] + incl - v;
  *total = ws[32];
  __syncthreads();
  return r;
}

__device__ __forceinline__ int block_sum(int v, int* ws) {
  int tot;
  block_exclusive_scan(v, ws, &tot);
  return tot;
}

// ------------------------------------------------------------- mbarriers --
__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* b, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(su32(b)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// One poll that may suspend the thread in hardware until the phase completes
// or about hint_ns pass: a waiting warp then takes no issue slots from the
// warps that share its scheduler.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
// Waits for the phase of parity `parity` to complete; gives up after
// limit_ns (1 s by default) or when another thread of the grid gave up, and
// then records MOE_ERR_TIMEOUT in *err and returns false.  Each poll suspends
// for at most a quarter of the limit (and 1 ms), so the limit holds to within
// that.
static __device__ __noinline__ bool mbar_wait(uint64_t* b, uint32_t parity, int* err,
                                              uint64_t limit_ns = 1000000000ull) {
  if (mbar_test(b, parity)) return true;
  const uint64_t t0 = gtimer();
  const uint32_t hint = (uint32_t)(limit_ns / 4 < 1000000ull ? limit_ns / 4 : 1000000ull);
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(b, parity, hint)) return true;
    if (gtimer() - t0 > limit_ns) {
      atomicExch(err, MOE_ERR_TIMEOUT);
      return false;
    }
    if ((it & 15) == 0 && *(volatile int*)err == MOE_ERR_TIMEOUT) return false;
  }
}


// mbar_wait with the ready case inline (no call when the phase is complete).
__device__ __forceinline__ bool mbar_wait_fast(uint64_t* b, uint32_t parity, int* err) {
  return mbar_test(b, parity) || mbar_wait(b, parity, err);
}

// One-dimensional bulk copy global -> shared (16-byte aligned, size a multiple
// of 16), completing as transaction bytes on an mbarrier.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(su32(dst)),
      "l"(src), "r"(bytes), "r"(su32(bar))
      : "memory");
}

}  // namespace moe
