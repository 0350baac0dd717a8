// The FP4 grouped GEMM (gate/up with SwiGLU, then down) shared by the prefill
// entry point and the decode forward.  Implemented in expert_prefill.cu.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace moe {

// A run of one slot's (or the shared expert's) pairs in the decode forward's
// sorted order: begin is the first sorted position (routed) or token (shared).
struct Group {
  int pool, slot, begin, count;
};

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

// ------------------------------------------------ block-scaled decode GEMM --
// Decode batches on tcgen05.mma.kind::mxf8f6f4 (decode_mx8.cu): E2M1 weights
// straight from the slot pool, activations as E4M3 hi + lo with a power-of-two
// scale per 32 elements.  Groups of up to kMx8MaxRows tokens.
constexpr int kMx8MaxRows = 48;

// Activation and h operands, rows in the plan's sorted order (routed pairs at
// their sorted position, the shared expert's tokens at P + t).
struct Mx8Bufs {
  uint8_t* xhi;  // [rows][H] E4M3
  uint8_t* xlo;
  uint8_t* xsc;  // [rows][H / 32] E8M0
  uint8_t* hhi;  // [rows][I]
  uint8_t* hlo;
  uint8_t* hsc;  // [rows][I / 32]
};

bool mx8_supported(const moe_expert_views* v);
size_t mx8_bytes(int H, int I, int rows);
void mx8_carve(uint8_t* base, int H, int I, int rows, Mx8Bufs* b);
// rows: the operand buffers' rows (P + T with the shared expert's, else P).
// mode 0: gate/up over the plan's groups (hdr, groups, perm; hdr[2 + mode] is the
// item counter, zeroed by the plan) -> h operands in b;
// mode 1: down -> o rows (pair index, or P + token for the shared expert).
moe_status mx8_gemm(const moe_expert_views* v, int mode, int T, int k, bool shared, int max_groups, int rows,
                    int* hdr, const Group* groups, const int* perm, const Mx8Bufs& b, float* o,
                    int32_t* d_error, cudaStream_t stream);

}  // namespace moe
