// Host side of the C ABI: error reporting, the slot-cache handle, the miss
// copies from the pinned host bank, and the load-time self test.
//
// The cache mirrors "Running DeepSeek-V4-Flash across four free GPUs",
// section "What the expert cache actually does": expert banks in pinned host
// RAM, a fixed number of VRAM slots, only the misses cross to the GPU.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"

namespace moe {

static thread_local std::string g_err;

moe_status fail(moe_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

moe_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MOE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

void clear_error() { g_err.clear(); }

// ------------------------------------------------------------- profiling --
struct ProfRec {
  int kernel;
  cudaEvent_t start, stop;
};
static std::mutex g_prof_mu;
static bool g_prof_on = false;
static std::vector<ProfRec> g_prof;
static std::vector<cudaEvent_t> g_prof_pool;

static cudaEvent_t prof_event() {
  if (!g_prof_pool.empty()) {
    cudaEvent_t e = g_prof_pool.back();
    g_prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

ProfScope::ProfScope(int kernel, cudaStream_t s) : k_(kernel), s_(s), stop_(nullptr) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on) return;
  cudaEvent_t a = prof_event(), b = prof_event();
  if (!a || !b) return;
  cudaEventRecord(a, s);
  g_prof.push_back({kernel, a, b});
  stop_ = b;
}

ProfScope::~ProfScope() {
  if (stop_) cudaEventRecord((cudaEvent_t)stop_, s_);
}

size_t fp4_bytes(int H, int I) {
  if (H <= 0 || I <= 0 || H % 32 || I % 32) return 0;
  size_t h = (size_t)H, i = (size_t)I;
  return 3 * (h * i / 2 + h * i / 32);
}
size_t int2_bytes(int H, int I) {
  if (H <= 0 || I <= 0 || H % 32 || I % 32) return 0;
  size_t h = (size_t)H, i = (size_t)I;
  return 3 * (h * i / 4 + h * i / 32);
}
size_t fp8_bytes(int H, int I) {
  if (H <= 0 || I <= 0 || H % 32 || I % 32) return 0;
  size_t h = (size_t)H, i = (size_t)I;
  return 3 * h * i + (2 * i + h) * 4;
}

__global__ void cache_reset_kernel(CacheDev c) {
  const int n = c.L * c.E;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    c.key_to_slot[i] = -1;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < c.S; i += gridDim.x * blockDim.x) {
    c.slot_key[i] = -1;
    c.slot_stamp[i] = 0;
  }
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    c.freq[i] = 0;
    c.freq_epoch[i] = 0;
  }
  if (c.R > 0) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) c.stage_of[i] = -1;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < c.R; i += gridDim.x * blockDim.x) c.stage_key[i] = -1;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *c.clock = 0;
    *c.calls = 0;
    if (c.R > 0) *c.stage_pos = 0;
  }
}

// Staging ring: predicted experts that are neither resident nor staged take
// ring slots round-robin (displacing older guesses, never a resident expert);
// the copy list (key, S + j) of the guesses that keep their slot is written
// for moe_copy_missing_device.  Ids are
// checked first; any id >= E makes the call a no-op with count -MOE_ERR_INVALID.
__global__ void prefetch_kernel(CacheDev c, int layer, const int32_t* experts, int n, int32_t* list_key,
                                int32_t* list_slot, int32_t* list_count) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  for (int i = 0; i < n; ++i)
    if (experts[i] >= c.E) {
      *list_count = -MOE_ERR_INVALID;
      return;
    }
  int m = 0;
  for (int i = 0; i < n; ++i) {
    const int e = experts[i];
    if (e < 0) continue;
    bool dup = false;
    for (int q = 0; q < i; ++q) dup = dup || experts[q] == e;
    if (dup) continue;
    const int key = layer * c.E + e;
    if (c.key_to_slot[key] >= 0 || c.stage_of[key] >= 0) continue;
    const uint32_t p = *c.stage_pos;
    const int j = (int)(p % (uint32_t)c.R);
    *c.stage_pos = p + 1;
    const int old = c.stage_key[j];
    if (old >= 0) c.stage_of[old] = -1;
    c.stage_key[j] = key;
    c.stage_of[key] = j;
    list_key[m] = key;
    list_slot[m] = c.S + j;
    ++m;
  }
  // assignments are round-robin, so only the last R of the call still hold
  // their ring slot: earlier ones were displaced within the call and are not
  // copied (two copies into one slot would race in the copy kernel)
  const int keep = m < c.R ? m : c.R;
  for (int q = 0; q < keep; ++q) {
    list_key[q] = list_key[m - keep + q];
    list_slot[q] = list_slot[m - keep + q];
  }
  *list_count = keep;
}

__global__ void cache_mark_empty_kernel(CacheDev c, int slot) {
  int key = c.slot_key[slot];
  if (key >= 0) c.key_to_slot[key] = -1;
  c.slot_key[slot] = -1;
}

// Copies the listed misses with GPU loads of the pinned bank (over the
// host-device link) and stores into the slots; reads the miss list and count
// on the device, so it needs no host round trip.  16-byte units, four loads in
// flight per thread before their stores.
// Bytes [b0, b0 + 16 * per) of each listed expert, one 16-byte unit per step.
template <typename Idx>
__device__ __forceinline__ void copy_units(const CacheDev& c, const uint8_t* bank, uint8_t* slots, size_t B,
                                           size_t b0, Idx per, const int32_t* miss_key, const int32_t* miss_slot,
                                           Idx total, int32_t* err) {
  const Idx stride = (Idx)gridDim.x * blockDim.x;
  const int K = c.L * c.E;
  for (Idx u0 = (Idx)blockIdx.x * blockDim.x + threadIdx.x; u0 < total; u0 += 4 * stride) {
    uint4 v[4];
    size_t dst[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const Idx u = u0 + (Idx)j * stride;
      dst[j] = (size_t)-1;
      if (u < total) {
        const int m = (int)(u / per);
        const size_t off = b0 + (size_t)(u - (Idx)m * per) * 16;
        const int key = miss_key[m], sl = miss_slot[m];
        if (key >= 0 && key < K && sl >= 0 && sl < c.S + c.R) {
          // a cache slot filled with a staged key copies from its staging slot
          const int st = (c.R > 0 && sl < c.S) ? c.stage_of[key] : -1;
          const uint8_t* src = st >= 0 ? slots + (size_t)(c.S + st) * B : bank + (size_t)key * B;
          v[j] = __ldcs(reinterpret_cast<const uint4*>(src + off));
          dst[j] = (size_t)sl * B + off;
        } else if (err && u - (Idx)m * per == 0) {
          // an entry that names no key or no slot is not copied; the slot it
          // was meant for holds stale bytes, so the call's status says so
          atomicCAS(err, 0, MOE_ERR_INVALID);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (dst[j] != (size_t)-1) *reinterpret_cast<uint4*>(slots + dst[j]) = v[j];
  }
}

// Copies the listed misses with GPU loads of the pinned bank (over the
// host-device link) and stores into the slots; reads the miss list and count
// on the device, so it needs no host round trip.  16-byte units, four loads in
// flight per thread before their stores.
// Part `part` of `parts` takes the list entries [n * part / parts, n * (part + 1) / parts),
// and of each expert the bytes [b0, b1) (16-byte multiples).
__global__ void __launch_bounds__(256) copy_missing_kernel(CacheDev c, const uint8_t* bank, uint8_t* slots,
                                                           size_t B, const int32_t* miss_key,
                                                           const int32_t* miss_slot, const int32_t* miss_count,
                                                           int part, int parts, size_t b0, size_t b1, int32_t* err) {
  const int n = *miss_count;
  if (n <= 0) return;
  const int m0 = (int)((long long)n * part / parts), m1 = (int)((long long)n * (part + 1) / parts);
  if (m1 <= m0) return;
  const size_t per = (b1 - b0) / 16;
  const size_t total = (size_t)(m1 - m0) * per;
  if (total < 0xFFFFFFFFull)
    copy_units<uint32_t>(c, bank, slots, B, b0, (uint32_t)per, miss_key + m0, miss_slot + m0, (uint32_t)total,
                         err);
  else
    copy_units<size_t>(c, bank, slots, B, b0, per, miss_key + m0, miss_slot + m0, total, err);
}

// One 16-byte load per `stride` bytes of the mapped bank (a page of it), so
// the GPU has translated every page before a miss copy reads it.  The loads
// bypass the caches; their xor feeds a store the compiler cannot drop.
__device__ uint32_t g_prime_sink;
__global__ void __launch_bounds__(256) prime_bank_kernel(const uint8_t* bank, size_t bytes, size_t stride) {
  uint32_t acc = 0;
  const size_t n = bytes / stride;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const uint4 v = __ldcv(reinterpret_cast<const uint4*>(bank + i * stride));
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (acc == 0x9e3779b9u) g_prime_sink = acc;  // rarely taken; keeps the loads
}

// One thread waits on an mbarrier that nothing arrives on; the bounded wait
// gives up after limit_ns and reports MOE_ERR_TIMEOUT (the same wait every
// pipelined kernel of this library uses).
__global__ void timeout_probe_kernel(uint64_t limit_ns, int32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    *status = 0;
    const bool ok = mbar_wait(&bar, 0, status, limit_ns);
    if (ok) *status = -1;  // cannot happen: nothing arrives
  }
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_last_error(void) { return g_err.c_str(); }
int moe_version(void) { return 1; }

size_t moe_fp4_expert_bytes(int H, int I) { return fp4_bytes(H, I); }
size_t moe_int2_expert_bytes(int H, int I) { return int2_bytes(H, I); }
size_t moe_fp8_expert_bytes(int H, int I) { return fp8_bytes(H, I); }

moe_status moe_cache_create(int num_slots, int num_layers, int num_experts, size_t expert_bytes,
                            void* d_slots, const void* h_bank, moe_cache** out) {
  clear_error();
  MOE_ARG(out != nullptr, "out is null");
  *out = nullptr;
  MOE_ARG(num_slots >= 1, "num_slots must be >= 1 (got %d)", num_slots);
  MOE_ARG(num_layers >= 1 && num_experts >= 1, "num_layers and num_experts must be >= 1");
  MOE_ARG(num_experts <= 4096, "num_experts must be <= 4096");
  MOE_ARG((long long)num_layers * num_experts < (1LL << 30), "too many keys");
  MOE_ARG(expert_bytes > 0 && expert_bytes % 16 == 0, "expert_bytes must be a positive multiple of 16");
  MOE_ARG(d_slots != nullptr, "d_slots is null");
  MOE_ARG(((uintptr_t)d_slots & 15) == 0, "d_slots must be 16-byte aligned");
  cudaPointerAttributes pa;
  MOE_CUDA(cudaPointerGetAttributes(&pa, d_slots));
  MOE_ARG(pa.type == cudaMemoryTypeDevice || pa.type == cudaMemoryTypeManaged,
          "d_slots is not device memory");
  if (h_bank != nullptr) {
    cudaPointerAttributes hb;
    MOE_CUDA(cudaPointerGetAttributes(&hb, h_bank));
    MOE_ARG(hb.type == cudaMemoryTypeHost,
            "h_bank is not page-locked host memory (allocate it pinned or register it)");
  }
  int dev = 0;
  MOE_CUDA(cudaGetDevice(&dev));
  const size_t S = (size_t)num_slots, K = (size_t)num_layers * num_experts;
  const size_t bytes = S * 8 + 8 + 8 + S * 4 + K * 4 + K * 8 + 64;
  void* state = nullptr;
  cudaError_t e = cudaMalloc(&state, bytes);
  if (e != cudaSuccess) return fail(MOE_ERR_NOMEM, "cudaMalloc of %zu bytes of cache state: %s", bytes,
                                    cudaGetErrorString(e));
  moe_cache* c = new moe_cache();
  c->S = num_slots;
  c->L = num_layers;
  c->E = num_experts;
  c->B = expert_bytes;
  c->d_slots = (uint8_t*)d_slots;
  c->h_bank = (const uint8_t*)h_bank;
  c->d_state = state;
  c->device = dev;
  c->fail_copy_index = -1;
  c->bank_dev = nullptr;
  if (h_bank != nullptr) {
    void* dp = nullptr;
    if (cudaHostGetDevicePointer(&dp, const_cast<void*>(h_bank), 0) == cudaSuccess)
      c->bank_dev = (const uint8_t*)dp;
    else
      cudaGetLastError();  // not mapped: moe_copy_missing_device is unavailable for this cache
  }
  uint8_t* p = (uint8_t*)state;
  c->dev.slot_stamp = (uint64_t*)p;
  p += S * 8;
  c->dev.clock = (uint64_t*)p;
  p += 8;
  c->dev.slot_key = (int32_t*)p;
  p += S * 4;
  c->dev.key_to_slot = (int32_t*)p;
  p += K * 4;
  c->dev.freq = (uint32_t*)p;
  p += K * 4;
  c->dev.freq_epoch = (uint32_t*)p;
  p += K * 4;
  c->dev.calls = (uint64_t*)(((uintptr_t)p + 7) & ~(uintptr_t)7);
  c->dev.policy = MOE_EVICT_LRU;
  c->dev.decay_calls = 1;
  c->dev.R = 0;
  c->dev.stage_key = nullptr;
  c->dev.stage_of = nullptr;
  c->dev.stage_pos = nullptr;
  c->d_stage = nullptr;
  c->dev.S = num_slots;
  c->dev.L = num_layers;
  c->dev.E = num_experts;
  cache_reset_kernel<<<64, 256>>>(c->dev);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(state);
    delete c;
    return cuda_fail(e, "cache reset");
  }
  *out = c;
  return MOE_OK;
}

moe_status moe_cache_destroy(moe_cache* c) {
  clear_error();
  if (c == nullptr) return MOE_OK;
  cudaError_t e = cudaFree(c->d_state);
  if (c->d_stage) cudaFree(c->d_stage);
  delete c;
  if (e != cudaSuccess) return cuda_fail(e, "cudaFree(cache state)");
  return MOE_OK;
}

moe_status moe_cache_reset(moe_cache* c, cudaStream_t s) {
  clear_error();
  MOE_ARG(c != nullptr, "cache is null");
  cache_reset_kernel<<<64, 256, 0, s>>>(c->dev);
  return check_launch("cache_reset_kernel");
}

moe_status moe_cache_state(moe_cache* c, int32_t** slot_key, uint64_t** slot_stamp,
                           int32_t** key_to_slot, uint64_t** clock) {
  clear_error();
  MOE_ARG(c != nullptr, "cache is null");
  if (slot_key) *slot_key = c->dev.slot_key;
  if (slot_stamp) *slot_stamp = c->dev.slot_stamp;
  if (key_to_slot) *key_to_slot = c->dev.key_to_slot;
  if (clock) *clock = c->dev.clock;
  return MOE_OK;
}

moe_status moe_cache_export(moe_cache* c, int32_t* h_slot_key, uint64_t* h_slot_stamp,
                            uint64_t* h_clock) {
  clear_error();
  MOE_ARG(c != nullptr && h_slot_key && h_slot_stamp && h_clock, "null argument");
  MOE_CUDA(cudaDeviceSynchronize());
  MOE_CUDA(cudaMemcpy(h_slot_key, c->dev.slot_key, (size_t)c->S * 4, cudaMemcpyDeviceToHost));
  MOE_CUDA(cudaMemcpy(h_slot_stamp, c->dev.slot_stamp, (size_t)c->S * 8, cudaMemcpyDeviceToHost));
  MOE_CUDA(cudaMemcpy(h_clock, c->dev.clock, 8, cudaMemcpyDeviceToHost));
  return MOE_OK;
}

moe_status moe_cache_import(moe_cache* c, const int32_t* h_slot_key, const uint64_t* h_slot_stamp,
                            uint64_t clock) {
  clear_error();
  MOE_ARG(c != nullptr && h_slot_key && h_slot_stamp, "null argument");
  const int K = c->L * c->E;
  std::vector<int32_t> k2s((size_t)K, -1);
  std::vector<uint64_t> seen;
  for (int s = 0; s < c->S; ++s) {
    int key = h_slot_key[s];
    if (key < 0) continue;
    MOE_ARG(key < K, "slot %d holds key %d >= L*E", s, key);
    MOE_ARG(k2s[key] < 0, "key %d held by two slots", key);
    MOE_ARG(h_slot_stamp[s] < clock, "slot %d has a stamp not below the clock", s);
    k2s[key] = s;
    seen.push_back(h_slot_stamp[s]);
  }
  std::sort(seen.begin(), seen.end());
  for (size_t i = 1; i < seen.size(); ++i) MOE_ARG(seen[i] != seen[i - 1], "duplicate stamps");
  MOE_CUDA(cudaDeviceSynchronize());
  MOE_CUDA(cudaMemcpy(c->dev.slot_key, h_slot_key, (size_t)c->S * 4, cudaMemcpyHostToDevice));
  MOE_CUDA(cudaMemcpy(c->dev.slot_stamp, h_slot_stamp, (size_t)c->S * 8, cudaMemcpyHostToDevice));
  MOE_CUDA(cudaMemcpy(c->dev.key_to_slot, k2s.data(), (size_t)K * 4, cudaMemcpyHostToDevice));
  MOE_CUDA(cudaMemcpy(c->dev.clock, &clock, 8, cudaMemcpyHostToDevice));
  return MOE_OK;
}

moe_status moe_cache_set_policy(moe_cache* c, int policy, int decay_calls) {
  clear_error();
  MOE_ARG(c != nullptr, "cache is null");
  MOE_ARG(policy == MOE_EVICT_LRU || policy == MOE_EVICT_LFU, "policy must be MOE_EVICT_LRU or MOE_EVICT_LFU");
  MOE_ARG(decay_calls >= 1, "decay_calls must be >= 1");
  c->dev.policy = policy;
  c->dev.decay_calls = decay_calls;
  return MOE_OK;
}

moe_status moe_cache_seed_frequency(moe_cache* c, const uint32_t* h_counts) {
  clear_error();
  MOE_ARG(c != nullptr && h_counts != nullptr, "null argument");
  const size_t K = (size_t)c->L * c->E;
  MOE_CUDA(cudaDeviceSynchronize());
  uint64_t calls = 0;
  MOE_CUDA(cudaMemcpy(&calls, c->dev.calls, 8, cudaMemcpyDeviceToHost));
  const uint32_t epoch = (uint32_t)(calls / (uint64_t)c->dev.decay_calls);
  std::vector<uint32_t> cnt(K), ep(K, epoch);
  for (size_t i = 0; i < K; ++i) cnt[i] = h_counts[i] < kFreqCap ? h_counts[i] : kFreqCap;
  MOE_CUDA(cudaMemcpy(c->dev.freq, cnt.data(), K * 4, cudaMemcpyHostToDevice));
  MOE_CUDA(cudaMemcpy(c->dev.freq_epoch, ep.data(), K * 4, cudaMemcpyHostToDevice));
  return MOE_OK;
}

moe_status moe_cache_export_frequency(moe_cache* c, uint32_t* h_counts, uint32_t* h_epochs, uint64_t* h_calls) {
  clear_error();
  MOE_ARG(c != nullptr && h_counts && h_epochs && h_calls, "null argument");
  const size_t K = (size_t)c->L * c->E;
  MOE_CUDA(cudaDeviceSynchronize());
  MOE_CUDA(cudaMemcpy(h_counts, c->dev.freq, K * 4, cudaMemcpyDeviceToHost));
  MOE_CUDA(cudaMemcpy(h_epochs, c->dev.freq_epoch, K * 4, cudaMemcpyDeviceToHost));
  MOE_CUDA(cudaMemcpy(h_calls, c->dev.calls, 8, cudaMemcpyDeviceToHost));
  return MOE_OK;
}

moe_status moe_cache_set_staging(moe_cache* c, int num_stage) {
  clear_error();
  MOE_ARG(c != nullptr, "cache is null");
  MOE_ARG(num_stage >= 0 && num_stage <= 65536, "num_stage out of [0, 65536]");
  MOE_CUDA(cudaDeviceSynchronize());
  if (c->d_stage) {
    MOE_CUDA(cudaFree(c->d_stage));
    c->d_stage = nullptr;
  }
  c->dev.R = 0;
  c->dev.stage_key = c->dev.stage_of = nullptr;
  c->dev.stage_pos = nullptr;
  if (num_stage == 0) return MOE_OK;
  const size_t K = (size_t)c->L * c->E;
  const size_t bytes = (size_t)num_stage * 4 + K * 4 + 16;
  void* p = nullptr;
  cudaError_t e = cudaMalloc(&p, bytes);
  if (e != cudaSuccess) return fail(MOE_ERR_NOMEM, "cudaMalloc of %zu bytes of staging state: %s", bytes,
                                    cudaGetErrorString(e));
  c->d_stage = p;
  c->dev.R = num_stage;
  c->dev.stage_key = (int32_t*)p;
  c->dev.stage_of = (int32_t*)p + num_stage;
  c->dev.stage_pos = (uint32_t*)((int32_t*)p + num_stage + K);
  MOE_CUDA(cudaMemset(c->dev.stage_key, 0xff, (size_t)num_stage * 4));
  MOE_CUDA(cudaMemset(c->dev.stage_of, 0xff, K * 4));
  MOE_CUDA(cudaMemset(c->dev.stage_pos, 0, 4));
  MOE_CUDA(cudaDeviceSynchronize());
  return MOE_OK;
}

moe_status moe_prefetch(moe_cache* c, int layer_id, const int32_t* d_experts, int n, int32_t* d_list_key,
                        int32_t* d_list_slot, int32_t* d_list_count, cudaStream_t stream) {
  clear_error();
  MOE_ARG(c != nullptr, "cache is null");
  MOE_ARG(c->dev.R > 0, "the cache has no staging ring (moe_cache_set_staging)");
  MOE_ARG(layer_id >= 0 && layer_id < c->L, "layer_id %d out of [0, %d)", layer_id, c->L);
  MOE_ARG(n >= 0 && n <= 4096, "n out of [0, 4096]");
  MOE_ARG(d_list_count && (n == 0 || (d_experts && d_list_key && d_list_slot)), "null pointer");
  prefetch_kernel<<<1, 32, 0, stream>>>(c->dev, layer_id, d_experts, n, d_list_key, d_list_slot, d_list_count);
  return check_launch("prefetch_kernel");
}

moe_status moe_cache_export_staging(moe_cache* c, int32_t* h_stage_key, uint32_t* h_pos) {
  clear_error();
  MOE_ARG(c != nullptr && h_stage_key && h_pos, "null argument");
  MOE_ARG(c->dev.R > 0, "the cache has no staging ring");
  MOE_CUDA(cudaDeviceSynchronize());
  MOE_CUDA(cudaMemcpy(h_stage_key, c->dev.stage_key, (size_t)c->dev.R * 4, cudaMemcpyDeviceToHost));
  MOE_CUDA(cudaMemcpy(h_pos, c->dev.stage_pos, 4, cudaMemcpyDeviceToHost));
  return MOE_OK;
}

moe_status moe_cache_prime_bank(moe_cache* c, cudaStream_t stream) {
  clear_error();
  MOE_ARG(c != nullptr, "cache is null");
  MOE_ARG(c->bank_dev != nullptr, "the host bank is not mapped into the device address space");
  MOE_ARG(((uintptr_t)c->bank_dev & 15) == 0, "the host bank must be 16-byte aligned");
  const size_t bytes = (size_t)c->L * c->E * c->B;
  int dev = 0, sms = 1;
  MOE_CUDA(cudaGetDevice(&dev));
  MOE_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  prime_bank_kernel<<<sms * 4, 256, 0, stream>>>(c->bank_dev, bytes, 4096);
  return check_launch("prime_bank_kernel");
}

static moe_status copy_missing_launch(moe_cache* c, const int32_t* d_miss_key, const int32_t* d_miss_slot,
                                      const int32_t* d_miss_count, int part, int n_parts, size_t b0, size_t b1,
                                      int max_ctas, int32_t* d_error, cudaStream_t stream) {
  MOE_ARG(c != nullptr, "cache is null");
  MOE_ARG(d_miss_key && d_miss_slot && d_miss_count, "null miss list");
  MOE_ARG(c->bank_dev != nullptr, "the host bank is not mapped into the device address space");
  MOE_ARG(c->B % 16 == 0, "expert bytes %zu not a multiple of 16", c->B);
  MOE_ARG(((uintptr_t)c->bank_dev & 15) == 0 && ((uintptr_t)c->d_slots & 15) == 0,
          "the host bank and the slot pool must be 16-byte aligned");
  MOE_ARG(n_parts >= 1 && n_parts <= MOE_MAX_COPY_PARTS && part >= 0 && part < n_parts,
          "part %d of %d: need 0 <= part < n_parts <= %d", part, n_parts, MOE_MAX_COPY_PARTS);
  MOE_ARG(b0 < b1 && b1 <= c->B && b0 % 16 == 0 && b1 % 16 == 0,
          "byte range [%zu, %zu) not within [0, %zu) in 16-byte units", b0, b1, c->B);
  MOE_ARG(max_ctas >= 0, "max_ctas < 0");
  int dev = 0, sms = 1;
  MOE_CUDA(cudaGetDevice(&dev));
  MOE_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  ProfScope ps(MOE_K_COPY, stream);
  const int grid = max_ctas > 0 && max_ctas < sms * 4 ? max_ctas : sms * 4;
  copy_missing_kernel<<<grid, 256, 0, stream>>>(c->dev, c->bank_dev, c->d_slots, c->B, d_miss_key, d_miss_slot,
                                                  d_miss_count, part, n_parts, b0, b1, d_error);
  return check_launch("copy_missing_kernel");
}

moe_status moe_copy_missing_device_part(moe_cache* c, const int32_t* d_miss_key, const int32_t* d_miss_slot,
                                        const int32_t* d_miss_count, int part, int n_parts, int max_ctas,
                                        int32_t* d_error, cudaStream_t stream) {
  clear_error();
  MOE_ARG(c != nullptr, "cache is null");
  return copy_missing_launch(c, d_miss_key, d_miss_slot, d_miss_count, part, n_parts, 0, c->B, max_ctas, d_error,
                             stream);
}

moe_status moe_copy_missing_device_slice(moe_cache* c, const int32_t* d_miss_key, const int32_t* d_miss_slot,
                                         const int32_t* d_miss_count, int part, int n_parts, size_t byte_begin,
                                         size_t byte_end, int max_ctas, int32_t* d_error, cudaStream_t stream) {
  clear_error();
  return copy_missing_launch(c, d_miss_key, d_miss_slot, d_miss_count, part, n_parts, byte_begin, byte_end,
                             max_ctas, d_error, stream);
}

moe_status moe_copy_missing_device_range(moe_cache* c, const int32_t* d_miss_key, const int32_t* d_miss_slot,
                                         const int32_t* d_miss_count, size_t byte_begin, size_t byte_end,
                                         int max_ctas, int32_t* d_error, cudaStream_t stream) {
  clear_error();
  return copy_missing_launch(c, d_miss_key, d_miss_slot, d_miss_count, 0, 1, byte_begin, byte_end, max_ctas,
                             d_error, stream);
}

moe_status moe_copy_missing_device(moe_cache* c, const int32_t* d_miss_key, const int32_t* d_miss_slot,
                                   const int32_t* d_miss_count, int max_ctas, int32_t* d_error,
                                   cudaStream_t stream) {
  clear_error();
  MOE_ARG(c != nullptr, "cache is null");
  return copy_missing_launch(c, d_miss_key, d_miss_slot, d_miss_count, 0, 1, 0, c->B, max_ctas, d_error, stream);
}

moe_status moe_copy_layer(const void* h_bank, int layer_id, int num_experts, size_t expert_bytes, void* d_buf,
                          cudaStream_t stream) {
  clear_error();
  MOE_ARG(h_bank && d_buf, "null pointer");
  MOE_ARG(layer_id >= 0 && num_experts >= 1 && expert_bytes > 0, "bad layer, expert count or size");
  cudaPointerAttributes hb;
  MOE_CUDA(cudaPointerGetAttributes(&hb, h_bank));
  MOE_ARG(hb.type == cudaMemoryTypeHost, "h_bank is not page-locked host memory");
  const size_t bytes = (size_t)num_experts * expert_bytes;
  const uint8_t* src = (const uint8_t*)h_bank + (size_t)layer_id * bytes;
  MOE_CUDA(cudaMemcpyAsync(d_buf, src, bytes, cudaMemcpyHostToDevice, stream));
  return MOE_OK;
}

moe_status moe_debug_fail_copy(moe_cache* c, int index) {
  clear_error();
  MOE_ARG(c != nullptr, "cache is null");
  c->fail_copy_index = index;
  return MOE_OK;
}

moe_status moe_copy_missing(moe_cache* c, const int32_t* h_miss_key, const int32_t* h_miss_slot,
                            int n_miss, cudaStream_t copy_stream, cudaEvent_t ready,
                            cudaEvent_t done) {
  clear_error();
  MOE_ARG(c != nullptr, "cache is null");
  MOE_ARG(n_miss >= 0 && n_miss <= c->S, "n_miss %d out of [0, S]", n_miss);
  MOE_ARG(n_miss == 0 || (h_miss_key && h_miss_slot), "null miss list");
  MOE_ARG(n_miss == 0 || c->h_bank != nullptr, "cache has no host bank");
  const int K = c->L * c->E;
  for (int i = 0; i < n_miss; ++i) {
    MOE_ARG(h_miss_key[i] >= 0 && h_miss_key[i] < K, "miss %d: key %d out of range", i, h_miss_key[i]);
    MOE_ARG(h_miss_slot[i] >= 0 && h_miss_slot[i] < c->S, "miss %d: slot %d out of range", i,
            h_miss_slot[i]);
  }
  if (ready) MOE_CUDA(cudaStreamWaitEvent(copy_stream, ready, 0));
  int failed_at = -1;
  cudaError_t err = cudaSuccess;
  for (int i = 0; i < n_miss; ++i) {
    if (i == c->fail_copy_index) {
      failed_at = i;
      err = cudaErrorUnknown;
      break;
    }
    err = cudaMemcpyAsync(c->d_slots + (size_t)h_miss_slot[i] * c->B,
                          c->h_bank + (size_t)h_miss_key[i] * c->B, c->B, cudaMemcpyHostToDevice,
                          copy_stream);
    if (err != cudaSuccess) {
      failed_at = i;
      break;
    }
  }
  if (failed_at >= 0) {
    // roll back: the failed miss and every later one hold nothing
    for (int i = failed_at; i < n_miss; ++i)
      cache_mark_empty_kernel<<<1, 1, 0, copy_stream>>>(c->dev, h_miss_slot[i]);
    if (done) cudaEventRecord(done, copy_stream);
    return fail(MOE_ERR_CUDA, "copy of miss %d (key %d -> slot %d) failed: %s; %d slot(s) marked empty",
                failed_at, h_miss_key[failed_at], h_miss_slot[failed_at],
                c->fail_copy_index == failed_at ? "injected failure" : cudaGetErrorString(err),
                n_miss - failed_at);
  }
  if (done) MOE_CUDA(cudaEventRecord(done, copy_stream));
  return MOE_OK;
}

moe_status moe_profile_enable(int enable) {
  clear_error();
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (auto& r : g_prof) {
    g_prof_pool.push_back(r.start);
    g_prof_pool.push_back(r.stop);
  }
  g_prof.clear();
  g_prof_on = enable != 0;
  return MOE_OK;
}

moe_status moe_profile_query(int kernel, double* total_ms, int* launches) {
  clear_error();
  MOE_ARG(kernel >= 0 && kernel < MOE_K_COUNT && total_ms && launches, "bad arguments");
  std::lock_guard<std::mutex> lk(g_prof_mu);
  double t = 0.0;
  int n = 0;
  for (auto& r : g_prof) {
    if (r.kernel != kernel) continue;
    MOE_CUDA(cudaEventSynchronize(r.stop));
    float ms = 0.f;
    MOE_CUDA(cudaEventElapsedTime(&ms, r.start, r.stop));
    t += ms;
    ++n;
  }
  *total_ms = t;
  *launches = n;
  return MOE_OK;
}

moe_status moe_profile_timeline(int max, int32_t* kernel, double* start_ms, double* stop_ms, int* n) {
  clear_error();
  MOE_ARG(max >= 0 && kernel && start_ms && stop_ms && n, "bad arguments");
  std::lock_guard<std::mutex> lk(g_prof_mu);
  *n = (int)g_prof.size();
  for (int i = 0; i < (int)g_prof.size() && i < max; ++i) {
    const ProfRec& r = g_prof[i];
    MOE_CUDA(cudaEventSynchronize(r.stop));
    float a = 0.f, b = 0.f;
    MOE_CUDA(cudaEventElapsedTime(&a, g_prof[0].start, r.start));
    MOE_CUDA(cudaEventElapsedTime(&b, g_prof[0].start, r.stop));
    kernel[i] = r.kernel;
    start_ms[i] = a;
    stop_ms[i] = b;
  }
  return MOE_OK;
}

moe_status moe_debug_timeout_probe(int64_t limit_ns, int32_t* d_status, cudaStream_t stream) {
  clear_error();
  MOE_ARG(d_status != nullptr, "d_status is null");
  MOE_ARG(limit_ns > 0 && limit_ns <= 2000000000LL, "limit_ns must be in (0, 2e9]");
  timeout_probe_kernel<<<1, 32, 0, stream>>>((uint64_t)limit_ns, d_status);
  return check_launch("timeout_probe_kernel");
}

moe_status moe_selftest(void) {
  clear_error();
  // Router on one known row, then a two-slot cache round trip with copies.
  const int E = 4, k = 2, S = 2, B = 64;
  float h_logits[E] = {0.5f, -1.0f, 2.0f, 0.5f};
  float* d_logits = nullptr;
  int32_t* d_i = nullptr;  // ids[2], slots[2], miss_key[2], miss_slot[2], count, done
  float* d_w = nullptr;
  uint8_t* d_slots = nullptr;
  uint8_t* h_bank = nullptr;
  moe_cache* c = nullptr;
  moe_status st = MOE_OK;
  int32_t h_i[10];
  float h_w[2];
  uint8_t h_slot_bytes[S * B];
#define ST_CUDA(x)                                    \
  do {                                                \
    cudaError_t _e = (x);                             \
    if (_e != cudaSuccess) {                          \
      st = cuda_fail(_e, #x);                         \
      goto out;                                       \
    }                                                 \
  } while (0)
  ST_CUDA(cudaMalloc(&d_logits, sizeof h_logits));
  ST_CUDA(cudaMalloc(&d_i, sizeof h_i));
  ST_CUDA(cudaMalloc(&d_w, sizeof h_w));
  ST_CUDA(cudaMalloc(&d_slots, S * B));
  ST_CUDA(cudaHostAlloc(&h_bank, E * B, cudaHostAllocDefault));
  for (int i = 0; i < E * B; ++i) h_bank[i] = (uint8_t)(i * 7 + 1);
  ST_CUDA(cudaMemcpy(d_logits, h_logits, sizeof h_logits, cudaMemcpyHostToDevice));
  if ((st = moe_router_topk(d_logits, 1, E, k, 1, d_i, d_w, 0)) != MOE_OK) goto out;
  if ((st = moe_cache_create(S, 1, E, B, d_slots, h_bank, &c)) != MOE_OK) goto out;
  if ((st = moe_slot_ensure(c, 0, d_i, d_i + 2, 1, k, 0, k, MOE_FETCH, 0, d_i + 4, d_i + 6, d_i + 8,
                            d_i + 9, 0)) != MOE_OK)
    goto out;
  ST_CUDA(cudaMemcpy(h_i, d_i, sizeof h_i, cudaMemcpyDeviceToHost));
  ST_CUDA(cudaMemcpy(h_w, d_w, sizeof h_w, cudaMemcpyDeviceToHost));
  if (h_i[0] != 2 || h_i[1] != 0 || h_i[2] != 0 || h_i[3] != 1 || h_i[8] != 2 || h_i[9] != 1 ||
      h_i[4] != 2 || h_i[5] != 0 || h_i[6] != 0 || h_i[7] != 1 || !(h_w[0] > h_w[1]) ||
      h_w[0] + h_w[1] < 0.999f || h_w[0] + h_w[1] > 1.001f) {
    st = fail(MOE_ERR_CUDA, "selftest: router/ensure produced wrong results");
    goto out;
  }
  if ((st = moe_copy_missing(c, h_i + 4, h_i + 6, h_i[8], 0, nullptr, nullptr)) != MOE_OK) goto out;
  ST_CUDA(cudaMemcpy(h_slot_bytes, d_slots, S * B, cudaMemcpyDeviceToHost));
  if (memcmp(h_slot_bytes, h_bank + 2 * B, B) != 0 || memcmp(h_slot_bytes + B, h_bank, B) != 0) {
    st = fail(MOE_ERR_CUDA, "selftest: copied slot bytes differ from the bank");
    goto out;
  }
  {
    // a tiny layer: H = 64, I = 32, two FP4 experts whose codes are all 1.0 with
    // unit E8M0 scales, x = 1, router weights 1/4 and 3/4.  gate = up = 64 for
    // every feature, h = SiLU(64) * 64 = 4096 (SiLU(64) rounds to 64 in fp32),
    // every output 32 * 4096 = 2^17, exact at every step and in bf16.
    const int FH = 64, FI = 32, FT = 1, FK = 2;
    const size_t EB = fp4_bytes(FH, FI);
    std::vector<uint8_t> ex(2 * EB);
    size_t off = 0;
    for (int m = 0; m < 3; ++m) {
      const size_t n = (m == 2) ? FH : FI, kk = (m == 2) ? FI : FH;
      for (size_t i = 0; i < n * kk / 2; ++i) ex[off + i] = 0x22;          // E2M1 1.0, both nibbles
      for (size_t i = 0; i < n * kk / 32; ++i) ex[off + n * kk / 2 + i] = 127;  // E8M0 2^0
      off += n * kk / 2 + n * kk / 32;
    }
    memcpy(ex.data() + EB, ex.data(), EB);
    std::vector<uint16_t> xv(FH, (uint16_t)0x3f80);  // bf16 1.0
    const int32_t hslots[FK] = {0, 1};
    const float hw[FK] = {0.25f, 0.75f};
    moe_expert_views v{};
    v.H = FH;
    v.I = FI;
    v.fp4_num_slots = 2;
    const size_t wsb = moe_expert_forward_workspace(&v, FT, FK);
    uint8_t* d_ex = nullptr;
    uint8_t* d_ws = nullptr;
    uint16_t* d_x = nullptr;
    uint16_t* d_y = nullptr;
    int32_t* d_sl = nullptr;
    float* d_fw = nullptr;
    int32_t* d_err = nullptr;
    uint16_t hy[FH];
    int32_t herr = -1;
    cudaError_t e = cudaMalloc(&d_ex, 2 * EB);
    if (e == cudaSuccess) e = cudaMalloc(&d_ws, wsb);
    if (e == cudaSuccess) e = cudaMalloc(&d_x, FH * 2);
    if (e == cudaSuccess) e = cudaMalloc(&d_y, FH * 2);
    if (e == cudaSuccess) e = cudaMalloc(&d_sl, sizeof hslots);
    if (e == cudaSuccess) e = cudaMalloc(&d_fw, sizeof hw);
    if (e == cudaSuccess) e = cudaMalloc(&d_err, sizeof herr);
    if (e == cudaSuccess) e = cudaMemcpy(d_ex, ex.data(), 2 * EB, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(d_x, xv.data(), FH * 2, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(d_sl, hslots, sizeof hslots, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(d_fw, hw, sizeof hw, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
      st = cuda_fail(e, "selftest: forward buffers");
    } else {
      v.fp4_slots = d_ex;
      st = moe_expert_forward(&v, d_x, FT, FK, d_sl, nullptr, d_fw, d_y, d_ws, wsb, d_err, 0);
      if (st == MOE_OK) {
        e = cudaMemcpy(hy, d_y, FH * 2, cudaMemcpyDeviceToHost);
        if (e == cudaSuccess) e = cudaMemcpy(&herr, d_err, sizeof herr, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) {
          st = cuda_fail(e, "selftest: forward read-back");
        } else {
          bool good = herr == 0;
          for (int i = 0; i < FH; ++i) good = good && hy[i] == 0x4800;  // bf16 2^17
          if (!good) st = fail(MOE_ERR_CUDA, "selftest: the tiny layer's output differs from 2^17");
        }
      }
    }
    cudaFree(d_ex);
    cudaFree(d_ws);
    cudaFree(d_x);
    cudaFree(d_y);
    cudaFree(d_sl);
    cudaFree(d_fw);
    cudaFree(d_err);
  }
out:
#undef ST_CUDA
  if (c) moe_cache_destroy(c);
  cudaFree(d_logits);
  cudaFree(d_i);
  cudaFree(d_w);
  cudaFree(d_slots);
  if (h_bank) cudaFreeHost(h_bank);
  return st;
}

}  // extern "C"
