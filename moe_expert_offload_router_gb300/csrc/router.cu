// Router: softmax over the E expert logits, top-k (ties to the lower id),
// renormalisation of the kept weights.
//
// "Running DeepSeek-V4-Flash across four free GPUs", section "What the expert
// cache actually does" (the router picks top_k experts per token and layer);
// "An elephant through a straw", section "Not all six experts matter equally"
// (one weight per selected expert, renormalised over the survivors).
//
// One warp per token.  Lane l holds logits l, l+32, ... in registers; each of
// the k rounds takes the warp-wide maximum of (logit, -id) with a butterfly of
// shuffles, so selection compares the fp32 logits exactly.  Weights are
// exp(l_j - l_max) over the sum of the kept (or of all E when not
// renormalising), reduced in a fixed shuffle order: deterministic.
#include <math.h>

#include "common.cuh"

namespace moe {

template <int VPL>
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ logits, int T,
                                                          int E, int k, int renorm,
                                                          int32_t* __restrict__ ids,
                                                          float* __restrict__ w) {
  pdl_launch_dependents();  // the slot ensure may set up meanwhile
  pdl_wait();               // launched early: the logits come from the previous work on the stream
  const int warp = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  const float* row = logits + (size_t)warp * E;
  float v[VPL];
  uint64_t taken = 0;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? __ldg(row + e) : -INFINITY;
    if (e >= E) taken |= 1ull << i;
  }
  float my_v = 0.f;
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      if (!((taken >> i) & 1ull) && (v[i] > bv || (v[i] == bv && e < bi))) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1ull << (bi >> 5);
    if (lane == j) {
      my_v = bv;
      my_id = bi;
    }
  }
  const float mx = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = lane < k ? expf(my_v - mx) : 0.f;
  float den;
  if (renorm) {
    den = ex;
  } else {
    den = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (lane + 32 * i < E) den += expf(v[i] - mx);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  if (lane < k) {
    ids[(size_t)warp * k + lane] = my_id;
    w[(size_t)warp * k + lane] = ex / den;
  }
}

template <int VPL>
static moe_status launch_router(const float* logits, int T, int E, int k, int renorm, int32_t* ids,
                                float* w, cudaStream_t s) {
  const int tpb = 256, tok_per_block = tpb / 32;
  const int blocks = (T + tok_per_block - 1) / tok_per_block;
  ProfScope ps(MOE_K_ROUTER, s);
  cudaError_t e = launch_pdl(router_topk_kernel<VPL>, dim3(blocks), dim3(tpb), 0, s, logits, T, E, k, renorm, ids, w);
  if (e != cudaSuccess) return cuda_fail(e, "router_topk_kernel");
  return check_launch("router_topk_kernel");
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_router_topk(const float* logits, int T, int E, int k, int renorm,
                                      int32_t* topk_ids, float* topk_w, cudaStream_t stream) {
  clear_error();
  MOE_ARG(T >= 0, "T must be >= 0");
  MOE_ARG(E >= 1 && E <= 2048, "E must be in [1, 2048] (got %d)", E);
  MOE_ARG(k >= 1 && k <= E && k <= 32, "k must be in [1, min(E, 32)] (got %d)", k);
  if (T == 0) return MOE_OK;
  MOE_ARG(logits && topk_ids && topk_w, "null pointer");
  const int vpl = (E + 31) / 32;
  if (vpl <= 1) return launch_router<1>(logits, T, E, k, renorm, topk_ids, topk_w, stream);
  if (vpl <= 2) return launch_router<2>(logits, T, E, k, renorm, topk_ids, topk_w, stream);
  if (vpl <= 4) return launch_router<4>(logits, T, E, k, renorm, topk_ids, topk_w, stream);
  if (vpl <= 8) return launch_router<8>(logits, T, E, k, renorm, topk_ids, topk_w, stream);
  if (vpl <= 16) return launch_router<16>(logits, T, E, k, renorm, topk_ids, topk_w, stream);
  if (vpl <= 32) return launch_router<32>(logits, T, E, k, renorm, topk_ids, topk_w, stream);
  return launch_router<64>(logits, T, E, k, renorm, topk_ids, topk_w, stream);
}
