// The FP4 grouped GEMM (gate/up with SwiGLU, then down) shared by the prefill
// entry point and the decode forward.  Implemented in expert_prefill.cu.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace moe {

struct PfItem {
  int slot, row0, count, pad;
};

// Buffers of one grouped-GEMM call (all device memory, caller-carved).
struct GgBufs {
  int* offsets;        // [S + 1]
  int* perm;           // [P] sorted position -> pair index
  PfItem* items;       // [S + P / 256 + 1]
  int* nitems;         // [1]
  int* cnt;            // grouping scratch
  uint16_t* xg;        // [P, H] bf16 gathered activations
  __half* xg16;        // [P, H] fp16 copy, each row scaled by 2^-xsig[row]
  int* xsig;           // [P]
  __nv_bfloat16* hs;   // [P, I] bf16 SwiGLU outputs
  float* o;            // [P, H] fp32 per-pair outputs (row = pair index t*k + j)
};

bool grouped_gemm_supported(const moe_expert_views* v);
size_t gg_index_bytes(int T, int k, int S);                   // offsets .. cnt, 256-aligned pieces
void gg_carve_index(uint8_t* base, int T, int k, int S, GgBufs* b);
// Writes o rows of every pair with 0 <= slot < S; other rows are untouched.
// Waits before the down GEMM, whose matrices may still be landing: with n
// events and a per-slot part index (device int8 [S], -1 = none), the down GEMM
// runs once per part q after ready[q], over the items of the slots of part q;
// with one event (or no part index) it waits on the last and runs once.
struct DownParts {
  int n = 0;
  const cudaEvent_t* ready = nullptr;
  const int8_t* slot_part = nullptr;
};
// mx_act != 0: x and h are quantised to MXFP4 (OCP MX, blocks of 32 along K) and
// the products run on their exact values.
moe_status grouped_gemm_fp4(const moe_expert_views* v, const uint16_t* x, int T, int k, const int32_t* slots,
                            const GgBufs& b, int32_t* d_error, cudaStream_t stream,
                            const DownParts& down = DownParts(), int mx_act = 0);
// The FP8 shared expert (v->shared) over all T tokens on the tensor cores:
// xs = fp16 activations [T, H], row t scaled by 2^-xsig[t]; hs = bf16 SwiGLU
// scratch [T, I]; writes o rows o_row0 .. o_row0 + T - 1 (fp32 [., H]).
moe_status grouped_gemm_shared_fp8(const moe_expert_views* v, const __half* xs, const int* xsig, int T,
                                   __nv_bfloat16* hs, float* o, int o_row0, int32_t* d_error,
                                   cudaStream_t stream);

}  // namespace moe
