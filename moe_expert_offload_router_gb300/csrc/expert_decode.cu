// Grouped expert MLP for decode-sized batches: gate/up GEMV + SwiGLU, down
// GEMV, and the router-weighted combine with the shared expert.
//
// "Running DeepSeek-V4-Flash across four free GPUs", section "What the expert
// cache actually does" (the grouped expert GEMM over the slot views);
// "An elephant through a straw", sections "43 graphs, 43 syncs" (grouped-GEMV
// expert kernels fired per layer) and "Rig, model & methodology" (MXFP4
// experts, a 2.25-bit copy with fp8 group scales, one shared expert).
//
// Structure (all launches on the caller's stream):
//   plan kernel   block 0 sorts the kept pairs by (pool, slot), stably, in
//                 shared memory (a counting sort over the slots; a bitonic
//                 sort of (pool, slot, pair) keys when the pools hold more
//                 than 4096 slots) and cuts each slot's run into groups of up
//                 to G tokens; blocks 1..T scale each token's activations by
//                 a power of two so the largest is in [1, 2) and store fp16.
//   gate/up       persistent; a work item is (group, 32-row tile).  The
//                 group's activations are staged in shared memory in the
//                 weight format's pairing; each warp streams gate row n and
//                 up row n with 128-bit loads (lane l takes 16-byte chunks
//                 l, l+32, ...), decodes two codes per instruction into
//                 fp16x2, accumulates each 32-weight block in fp16x2, scales
//                 the block sum in fp32, reduces across lanes with shuffles
//                 and writes h = SiLU(g) * u in fp32.
//   down          same over W2 with h staged the same way (per-pair scale).
//   combine       y_t = sum_j w_tj o_tj (rank order) + shared, fp32 -> bf16.
// fp16 block sums cannot overflow: |code| <= 6 (E2M1), 1.5 (2-bit), 448
// (E4M3) times |activation| < 2 times 32 (16 for E4M3) terms stays below 2^15.
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "grouped_gemm.cuh"
#include "mx.cuh"

namespace moe {

constexpr int kG = 8;             // tokens per group
constexpr int kFwdThreads = 256;  // 8 warps
constexpr int kRowsGateUp = 32;   // rows of w1/w3 per gate/up work item
constexpr int kRowsDown = 64;     // rows of w2 per down work item
constexpr int kMaxPlanPairs = 4096;
constexpr int kPlanBins = 4096;  // (pool, slot) bins of the plan's counting sort (FP4 slots, then 2-bit)
constexpr int kGemmMinPairs = 256;  // from here on the FP4 routed pairs take the tcgen05 grouped GEMM

// Decode batches up to this many tokens get the block-scaled GEMM's operand
// buffers in their workspace (its groups are cut at kMx8MaxRows rows, so any
// batch size works; the bound keeps the workspace of larger calls small).
constexpr int kMx8MaxTokens = 64;

struct FwdLayout {
  size_t hdr, perm, groups, xsig, xs, h, o, hs16, hsig, gg, mx8, total;
  bool gemm;     // the FP4 routed pairs may take the grouped GEMM
  bool mx8_ok;   // room for the block-scaled decode GEMM's operands
};

static inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static FwdLayout fwd_layout(const moe_expert_views* v, int T, int k) {
  const int H = v->H, I = v->I;
  const size_t P = (size_t)T * k;
  const size_t ng = P + (T + kG - 1) / kG + 1;
  FwdLayout L;
  size_t off = 0;
  L.hdr = off;
  off = align256(off + 256);
  L.perm = off;
  off = align256(off + P * 4);
  L.groups = off;
  off = align256(off + ng * sizeof(Group));
  L.xsig = off;
  off = align256(off + (size_t)T * 4);
  L.xs = off;
  off = align256(off + (size_t)T * H * 2);
  L.h = off;
  off = align256(off + (P + T) * (size_t)I * 4);
  L.o = off;
  off = align256(off + (P + T) * (size_t)H * 4);
  L.hs16 = off;  // fp16 copy of h for the warp-MMA down kernel
  off = align256(off + (P + T) * (size_t)I * 2);
  L.hsig = off;
  off = align256(off + (P + T) * 4);
  L.gemm = (long long)P >= kGemmMinPairs && grouped_gemm_supported(v);
  L.gg = off;
  if (L.gemm) off = align256(off + gg_index_bytes(T, k, v->fp4_num_slots));
  L.mx8_ok = T >= 2 && T <= kMx8MaxTokens && mx8_supported(v);
  L.mx8 = off;
  if (L.mx8_ok) off = align256(off + mx8_bytes(H, I, (int)P + T));
  L.total = off;
  return L;
}

struct FwdArgs {
  int H, I, T, k, P;
  const uint8_t* fp4;
  int n4;
  const uint8_t* int2;
  int n2;
  const uint8_t* shared;
  size_t b4, b2;  // bytes per expert
  const uint16_t* x;
  const int32_t* slots;
  const int8_t* tags;
  const float* w;
  uint16_t* y;
  int32_t* err;
  int routed_gemm;  // routed pairs are computed by the grouped GEMM, not by these kernels
  int gemv_skip;    // bit per pool: groups of these pools are left to the warp-MMA kernels
  int mma_group;    // tokens per group of those pools (kG for the others)
  // workspace
  int* hdr;
  int* perm;
  Group* groups;
  int* xsig;
  __half* xs;
  float* h;
  float* o;
  __half* hs16;  // h in fp16, row r scaled by 2^-hsig[r] (warp-MMA down kernel)
  int* hsig;
  // block-scaled decode GEMM: E4M3 hi/lo activation rows in sorted order and
  // their scale bytes, written by the plan (null: not this path)
  uint8_t* xhi;
  uint8_t* xlo;
  uint8_t* xsc;
};

// ------------------------------------------------------------------ decode --

__device__ __forceinline__ float e8m0_f32(uint32_t e) {
  // 2^(e-127): exponent field e for e >= 1; e = 0 is the subnormal 2^-127.
  return e ? __uint_as_float(e << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ void fp4_word_to_h2(uint32_t w, __half2* out) {
  uint32_t r0, r1, r2, r3;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(w));
  out[0] = *reinterpret_cast<__half2*>(&r0);
  out[1] = *reinterpret_cast<__half2*>(&r1);
  out[2] = *reinterpret_cast<__half2*>(&r2);
  out[3] = *reinterpret_cast<__half2*>(&r3);
}

__device__ __forceinline__ __half2 e4m3x2_to_h2(uint32_t two_bytes) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo;\n\tcvt.u16.u32 lo, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
      : "=r"(r)
      : "r"(two_bytes));
  return *reinterpret_cast<__half2*>(&r);
}

__device__ __forceinline__ void fp8_word_to_h2(uint32_t w, __half2* out) {
  out[0] = e4m3x2_to_h2(w & 0xffffu);
  out[1] = e4m3x2_to_h2(w >> 16);
}

// 16 two-bit codes (element i at bits 2i) -> 8 fp16x2 holding the levels
// (q - 1.5) of elements (i, i + 8): the code is placed in the mantissa of
// 512 (ulp 0.5, so 512 + q exactly), then 513.5 is subtracted.
__device__ __forceinline__ void int2_word_to_h2(uint32_t w, __half2* out) {
  const __half2 bias = __halves2half2(__ushort_as_half((unsigned short)0x6003),
                                      __ushort_as_half((unsigned short)0x6003));
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t sh = i == 0 ? (w << 1) : (w >> (2 * i - 1));
    const uint32_t v = (sh & 0x00060006u) | 0x60006000u;
    out[i] = __hsub2(*reinterpret_cast<const __half2*>(&v), bias);
  }
}

__device__ __forceinline__ float h2sum(__half2 a) {
  const float2 f = __half22float2(a);
  return f.x + f.y;
}

__device__ __forceinline__ void lds4(const uint4* p, __half2* x) {
  const uint4 v = *p;
  x[0] = *reinterpret_cast<const __half2*>(&v.x);
  x[1] = *reinterpret_cast<const __half2*>(&v.y);
  x[2] = *reinterpret_cast<const __half2*>(&v.z);
  x[3] = *reinterpret_cast<const __half2*>(&v.w);
}

// Physical 16-byte unit within a chunk for each format's activation layout
// (rotations that keep a quarter-warp's 128-bit shared loads conflict-free).
__device__ __forceinline__ int unit_fp4(int c, int s) { return c * 4 + ((s + (c >> 1)) & 3); }
__device__ __forceinline__ int unit_int2(int c, int s) { return c * 8 + ((s + c) & 7); }
__device__ __forceinline__ int unit_fp8(int c, int s) { return c * 2 + ((s + (c >> 2)) & 1); }

// --------------------------------------------------------- chunk processors --
// Each adds, for two rows (r0, r1) and every staged token, one 16-byte code
// chunk's contribution to the lane's fp32 accumulators.

template <int NT>
__device__ __forceinline__ void chunk_fp4(uint4 q0, uint32_t e0, uint4 q1, uint32_t e1, int c,
                                          const uint4* xs, int xstride, int ntok, float* a0,
                                          float* a1) {
  __half2 w0[16], w1[16];
  fp4_word_to_h2(q0.x, w0);
  fp4_word_to_h2(q0.y, w0 + 4);
  fp4_word_to_h2(q0.z, w0 + 8);
  fp4_word_to_h2(q0.w, w0 + 12);
  fp4_word_to_h2(q1.x, w1);
  fp4_word_to_h2(q1.y, w1 + 4);
  fp4_word_to_h2(q1.z, w1 + 8);
  fp4_word_to_h2(q1.w, w1 + 12);
  const float s0 = e8m0_f32(e0), s1 = e8m0_f32(e1);
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    {
      const uint4* xp = xs + (size_t)t * xstride;
      __half2 x[16];
#pragma unroll
      for (int s = 0; s < 4; ++s) lds4(xp + unit_fp4(c, s), x + 4 * s);
      __half2 p0 = __hmul2(w0[0], x[0]), q0a = __hmul2(w0[8], x[8]);
      __half2 p1 = __hmul2(w1[0], x[0]), q1a = __hmul2(w1[8], x[8]);
#pragma unroll
      for (int i = 1; i < 8; ++i) {
        p0 = __hfma2(w0[i], x[i], p0);
        q0a = __hfma2(w0[8 + i], x[8 + i], q0a);
        p1 = __hfma2(w1[i], x[i], p1);
        q1a = __hfma2(w1[8 + i], x[8 + i], q1a);
      }
      a0[t] = fmaf(h2sum(p0) + h2sum(q0a), s0, a0[t]);
      a1[t] = fmaf(h2sum(p1) + h2sum(q1a), s1, a1[t]);
    }
  }
}

template <int NT>
__device__ __forceinline__ void chunk_int2(uint4 q0, uint32_t e0, uint4 q1, uint32_t e1, int c,
                                           const uint4* xs, int xstride, int ntok, float* a0,
                                           float* a1) {
  // 64 weights: words 0-1 form scale block 0, words 2-3 block 1; one block at a time
  const float2 s0 = __half22float2(e4m3x2_to_h2(e0));
  const float2 s1 = __half22float2(e4m3x2_to_h2(e1));
#pragma unroll
  for (int blk = 0; blk < 2; ++blk) {
    __half2 w0[16], w1[16];
    int2_word_to_h2(blk ? q0.z : q0.x, w0);
    int2_word_to_h2(blk ? q0.w : q0.y, w0 + 8);
    int2_word_to_h2(blk ? q1.z : q1.x, w1);
    int2_word_to_h2(blk ? q1.w : q1.y, w1 + 8);
    const float sa = blk ? s0.y : s0.x, sb = blk ? s1.y : s1.x;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const uint4* xp = xs + (size_t)t * xstride;
      __half2 x[16];
#pragma unroll
      for (int s = 0; s < 4; ++s) lds4(xp + unit_int2(c, 4 * blk + s), x + 4 * s);
      __half2 pa = __hmul2(w0[0], x[0]), ra = __hmul2(w1[0], x[0]);
#pragma unroll
      for (int i = 1; i < 16; ++i) {
        pa = __hfma2(w0[i], x[i], pa);
        ra = __hfma2(w1[i], x[i], ra);
      }
      a0[t] = fmaf(h2sum(pa), sa, a0[t]);
      a1[t] = fmaf(h2sum(ra), sb, a1[t]);
    }
  }
}

template <int NT>
__device__ __forceinline__ void chunk_fp8(uint4 q0, uint4 q1, int c, const uint4* xs, int xstride,
                                          int ntok, float* a0, float* a1) {
  __half2 w0[8], w1[8];
  fp8_word_to_h2(q0.x, w0);
  fp8_word_to_h2(q0.y, w0 + 2);
  fp8_word_to_h2(q0.z, w0 + 4);
  fp8_word_to_h2(q0.w, w0 + 6);
  fp8_word_to_h2(q1.x, w1);
  fp8_word_to_h2(q1.y, w1 + 2);
  fp8_word_to_h2(q1.z, w1 + 4);
  fp8_word_to_h2(q1.w, w1 + 6);
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    {
      const uint4* xp = xs + (size_t)t * xstride;
      __half2 x[8];
      lds4(xp + unit_fp8(c, 0), x);
      lds4(xp + unit_fp8(c, 1), x + 4);
      __half2 p0 = __hmul2(w0[0], x[0]), p1 = __hmul2(w1[0], x[0]);
#pragma unroll
      for (int i = 1; i < 8; ++i) {
        p0 = __hfma2(w0[i], x[i], p0);
        p1 = __hfma2(w1[i], x[i], p1);
      }
      a0[t] += h2sum(p0);
      a1[t] += h2sum(p1);
    }
  }
}

// ------------------------------------------------------------- row dot pairs --
// Lane-partial dot products of two rows against the staged tokens.  K is the
// row length; KC > 0 is K known at compile time (loads of all the lane's
// chunks are issued before any is consumed).

template <int KC, int NT>
__device__ __forceinline__ void rows_fp4(const uint8_t* c0, const uint8_t* s0, const uint8_t* c1,
                                         const uint8_t* s1, int K, const uint4* xs, int ntok,
                                         float* a0, float* a1) {
  const int lane = threadIdx.x & 31;
  const int xstride = K / 8;
  if constexpr (KC > 0 && KC % 1024 == 0) {
    constexpr int CPL = KC / 1024;
    uint4 q0[CPL], q1[CPL];
    uint32_t e0[CPL], e1[CPL];
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int c = lane + 32 * i;
      q0[i] = ld_stream_v4(c0 + (size_t)c * 16);
      q1[i] = ld_stream_v4(c1 + (size_t)c * 16);
      e0[i] = __ldg(s0 + c);
      e1[i] = __ldg(s1 + c);
    }
#pragma unroll
    for (int i = 0; i < CPL; ++i) chunk_fp4<NT>(q0[i], e0[i], q1[i], e1[i], lane + 32 * i, xs, xstride, ntok, a0, a1);
  } else {
    const int nch = K / 32;
    for (int c = lane; c < nch; c += 32)
      chunk_fp4<NT>(ld_stream_v4(c0 + (size_t)c * 16), __ldg(s0 + c), ld_stream_v4(c1 + (size_t)c * 16),
                __ldg(s1 + c), c, xs, xstride, ntok, a0, a1);
  }
}

template <int KC, int NT>
__device__ __forceinline__ void rows_int2(const uint8_t* c0, const uint8_t* s0, const uint8_t* c1,
                                          const uint8_t* s1, int K, const uint4* xs, int ntok,
                                          float* a0, float* a1) {
  const int lane = threadIdx.x & 31;
  const int xstride = K / 8;
  const int nch = K / 64;
  auto sc = [](const uint8_t* p, int c) -> uint32_t {
    return (uint32_t)__ldg(p + 2 * c) | ((uint32_t)__ldg(p + 2 * c + 1) << 8);
  };
  if constexpr (KC > 0 && KC % 2048 == 0) {
    constexpr int CPL = KC / 2048;
    uint4 q0[CPL], q1[CPL];
    uint32_t e0[CPL], e1[CPL];
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int c = lane + 32 * i;
      q0[i] = ld_stream_v4(c0 + (size_t)c * 16);
      q1[i] = ld_stream_v4(c1 + (size_t)c * 16);
      e0[i] = sc(s0, c);
      e1[i] = sc(s1, c);
    }
#pragma unroll
    for (int i = 0; i < CPL; ++i) chunk_int2<NT>(q0[i], e0[i], q1[i], e1[i], lane + 32 * i, xs, xstride, ntok, a0, a1);
  } else {
    for (int c = lane; c < nch; c += 32)
      chunk_int2<NT>(ld_stream_v4(c0 + (size_t)c * 16), sc(s0, c), ld_stream_v4(c1 + (size_t)c * 16),
                 sc(s1, c), c, xs, xstride, ntok, a0, a1);
  }
}

template <int KC, int NT>
__device__ __forceinline__ void rows_fp8(const uint8_t* c0, const uint8_t* c1, int K, const uint4* xs,
                                         int ntok, float* a0, float* a1) {
  const int lane = threadIdx.x & 31;
  const int xstride = K / 8;
  const int nch = K / 16;
  if constexpr (KC > 0 && KC % 512 == 0) {
    constexpr int CPL = KC / 512;
    uint4 q0[CPL], q1[CPL];
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int c = lane + 32 * i;
      q0[i] = ld_stream_v4(c0 + (size_t)c * 16);
      q1[i] = ld_stream_v4(c1 + (size_t)c * 16);
    }
#pragma unroll
    for (int i = 0; i < CPL; ++i) chunk_fp8<NT>(q0[i], q1[i], lane + 32 * i, xs, xstride, ntok, a0, a1);
  } else {
    for (int c = lane; c < nch; c += 32)
      chunk_fp8<NT>(ld_stream_v4(c0 + (size_t)c * 16), ld_stream_v4(c1 + (size_t)c * 16), c, xs, xstride,
                ntok, a0, a1);
  }
}

template <int NT>
__device__ __forceinline__ void warp_allreduce(float* a) {
#pragma unroll
  for (int t = 0; t < NT; ++t) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a[t] += __shfl_xor_sync(0xffffffffu, a[t], o);
  }
}

// ------------------------------------------------------------ matrix views --
// Canonical byte offsets of matrix m (0 = w1 [I,H], 1 = w3 [I,H], 2 = w2 [H,I])
// inside one expert of each format.
struct MatView {
  const uint8_t* codes;
  const uint8_t* scales;  // FP4: E8M0 [N][K/32]; INT2: E4M3 [N][K/32]; FP8: fp32 [N]
  int N, K;
};

__device__ __forceinline__ MatView mat_view(int pool, const uint8_t* expert, int H, int I, int m) {
  const size_t hi = (size_t)H * I;
  MatView v;
  v.N = (m == 2) ? H : I;
  v.K = (m == 2) ? I : H;
  size_t per, cb;
  if (pool == MOE_POOL_FP4) {
    cb = hi / 2;
    per = cb + hi / 32;
  } else if (pool == MOE_POOL_INT2) {
    cb = hi / 4;
    per = cb + hi / 32;
  } else {
    cb = hi;
    per = 0;  // FP8 matrices differ in row-scale size; computed below
  }
  if (pool != MOE_POOL_SHARED) {
    v.codes = expert + per * m;
    v.scales = v.codes + cb;
  } else {
    const size_t w1 = hi + (size_t)I * 4;  // w1 and w3: codes [I,H] + scales [I]
    v.codes = expert + w1 * m;
    v.scales = v.codes + hi;
  }
  return v;
}

// ----------------------------------------------------------------- staging --
// Copy ntok activation rows (fp16, already scaled) into the format's layout.
// src_row(i) gives the fp16 row of staged token i.
template <typename SrcFn>
__device__ void stage_rows(int pool, int K, int ntok, SrcFn src_row, uint4* xs) {
  const int units = K / 8;  // 16-byte units per row
  for (int u = threadIdx.x; u < ntok * units; u += blockDim.x) {
    const int i = u / units, uu = u % units;
    const __half* src = src_row(i);
    uint4 v;
    if (pool == MOE_POOL_FP4) {
      const int c = uu >> 2, sl = ((uu & 3) - (c >> 1)) & 3;
      v = *reinterpret_cast<const uint4*>(src + c * 32 + sl * 8);
    } else if (pool == MOE_POOL_SHARED) {
      const int c = uu >> 1, sl = ((uu & 1) - (c >> 2)) & 1;
      v = *reinterpret_cast<const uint4*>(src + c * 16 + sl * 8);
    } else {
      const int c = uu >> 3, sl = ((uu & 7) - c) & 7;
      const int base = c * 64 + (sl >> 1) * 16 + (sl & 1) * 4;
      __half2 hh[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) hh[m] = __halves2half2(src[base + m], src[base + m + 8]);
      v = *reinterpret_cast<uint4*>(hh);
    }
    xs[(size_t)i * units + uu] = v;
  }
}

// --------------------------------------------------------------- plan kernel --

__device__ __forceinline__ float block_max(float v, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) red[wid] = v;
  __syncthreads();
  if (wid == 0) {
    float t = lane < nw ? red[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
    if (lane == 0) red[32] = t;
  }
  __syncthreads();
  const float r = red[32];
  __syncthreads();
  return r;
}

// Power-of-two exponent s with amax * 2^-s in [1, 2) (0 when amax is 0),
// at least -126 so that 2^s is a normal float for the epilogues that multiply
// it back (a smaller amax is scaled up by 2^126 only).
__device__ __forceinline__ int pow2_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  int e;
  frexpf(amax, &e);
  return max(-126, e - 1);
}

// Tokens per group: the warp-MMA kernels' pools take a.mma_group, the others kG.
__device__ __forceinline__ int group_size(const FwdArgs& a, int pool) {
  return (a.mma_group > 0 && pool >= 0 && pool < 31 && ((a.gemv_skip >> pool) & 1)) ? a.mma_group : kG;
}

// Sort key of pair p: (pool, slot, p) for a pair the kernels compute, ~0 for
// one they leave out (slot < 0 or a dropped tag), ~0 - 1 for a bad slot or tag.
__device__ __forceinline__ unsigned long long plan_key(const FwdArgs& a, int p) {
  const int sl = a.slots[p];
  const int tag = a.tags ? (int)a.tags[p] : MOE_TAG_FP4;
  if (sl < 0 || tag == MOE_TAG_DROP) return ~0ull;
  const int pool = tag == MOE_TAG_INT2 ? MOE_POOL_INT2 : MOE_POOL_FP4;
  const int npool = pool == MOE_POOL_FP4 ? a.n4 : a.n2;
  if ((tag == MOE_TAG_FP4 || tag == MOE_TAG_INT2) && sl < npool)
    return ((unsigned long long)((unsigned)pool << 30 | (unsigned)sl) << 32) | (unsigned)p;
  return ~0ull - 1;
}

// Token t's activations as E4M3 hi/lo with a power-of-two scale per 32
// elements (mx.cuh), written to the rows of its FP4 pairs in the sorted order
// (a pair's row is the number of kept keys below its own, the position the
// sort of block 0 gives it) and to row P + t for the shared expert.
__device__ void plan_mx8_rows(const FwdArgs& a, int t, int* dst, unsigned long long* keys) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // every pair's key, staged once in shared memory for the counts below
  for (int q = threadIdx.x; q < a.P; q += blockDim.x) keys[q] = plan_key(a, q);
  __syncthreads();
  for (int j = warp; j < a.k; j += (int)(blockDim.x >> 5)) {
    const int p = t * a.k + j;
    const unsigned long long key = keys[p];
    int below = 0;
    for (int q = lane; q < a.P; q += 32) below += keys[q] < key;
    below = __reduce_add_sync(0xffffffffu, below);
    if (lane == 0) dst[j] = (key < ~0ull - 1 && (key >> 62) == MOE_POOL_FP4) ? below : -1;
  }
  if (threadIdx.x == 0) dst[a.k] = a.shared ? a.P + t : -1;
  __syncthreads();
  const uint16_t* xr = a.x + (size_t)t * a.H;
  // 8 threads per 32-element block, 4 elements each (H is a multiple of 256,
  // so every warp is either whole or idle in each pass)
  for (int e0 = 4 * threadIdx.x; e0 < a.H; e0 += 4 * blockDim.x) {
    const uint2 raw = *reinterpret_cast<const uint2*>(xr + e0);
    float f[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u), __uint_as_float(raw.y << 16),
                  __uint_as_float(raw.y & 0xffff0000u)};
    float am = fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3])));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 4));
    const uint32_t sb = mx8_scale_byte(am);
    const float inv = __uint_as_float((254u - sb) << 23);
    uint32_t h01, l01, h23, l23;
    mx8_split2(f[0] * inv, f[1] * inv, h01, l01);
    mx8_split2(f[2] * inv, f[3] * inv, h23, l23);
    const uint32_t hw = h01 | (h23 << 16), lw = l01 | (l23 << 16);
    for (int d = 0; d <= a.k; ++d) {
      const int row = dst[d];
      if (row < 0) continue;
      *reinterpret_cast<uint32_t*>(a.xhi + (size_t)row * a.H + e0) = hw;
      *reinterpret_cast<uint32_t*>(a.xlo + (size_t)row * a.H + e0) = lw;
      if ((threadIdx.x & 7) == 0) a.xsc[(size_t)row * (a.H / 32) + e0 / 32] = (uint8_t)sb;
    }
  }
}

// After the routed groups: the shared expert's groups (runs of its group
// size over the tokens) and the header (one thread).
__device__ void plan_finish(const FwdArgs& a, int ngroups, bool bad) {
  int n = ngroups;
  if (a.shared) {
    const int gs = group_size(a, MOE_POOL_SHARED);
    for (int t0 = 0; t0 < a.T; t0 += gs) {
      Group g;
      g.pool = MOE_POOL_SHARED;
      g.slot = 0;
      g.begin = t0;
      g.count = min(gs, a.T - t0);
      a.groups[n++] = g;
    }
  }
  a.hdr[0] = n;
  a.hdr[1] = ngroups;
  a.hdr[2] = 0;  // work counters of the warp-MMA gate/up and down kernels
  a.hdr[3] = 0;
  if (a.err && bad) atomicCAS(a.err, 0, MOE_ERR_INVALID);  // the caller's call cleared it
}

// Block 0 of the plan when the (pool, slot) bins fit in shared memory: a
// stable counting sort.  Bin of a kept pair = its FP4 slot, or n4 + its 2-bit
// slot, so bin order is the (pool, slot) order; the bins' counts give each
// bin's first sorted position and its groups (runs cut every group-size
// pairs) directly, and one warp places the pairs 32 at a time in pair order
// (rank among equal bins by __match_any_sync), so that each bin keeps its
// pairs in increasing pair index: the order a sort on (pool, slot, pair)
// gives.
__device__ void plan_groups_counting(const FwdArgs& a, uint8_t* smem_raw) {
  int* cnt = reinterpret_cast<int*>(smem_raw);  // [kPlanBins] pairs per bin
  int* cur = cnt + kPlanBins;                   // [kPlanBins] next sorted position of each bin
  int* binv = cur + kPlanBins;                  // [kMaxPlanPairs] bin of each pair, -1 if left out
  int* ws = binv + kMaxPlanPairs;               // [34] scan workspace
  int* scal = ws + 34;
  const int P = a.P, nb = a.n4 + a.n2;
  const int tid = threadIdx.x, NT = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31;
  for (int b = tid; b < nb; b += NT) cnt[b] = 0;
  if (tid == 0) scal[0] = 0;
  __syncthreads();
  for (int p = tid; p < P; p += NT) {
    const unsigned long long key = plan_key(a, p);
    int b = -1;
    if (key == ~0ull - 1) {
      scal[0] = 1;
    } else if (key != ~0ull) {
      const int slot = (int)((key >> 32) & 0x3fffffffu);
      b = (key >> 62) == MOE_POOL_FP4 ? slot : a.n4 + slot;
      atomicAdd(&cnt[b], 1);
    }
    binv[p] = b;
  }
  __syncthreads();
  // each thread takes a run of bins: their pairs and groups, scanned over the block
  const int per = (nb + NT - 1) / NT;
  const int b0 = min(nb, tid * per), b1 = min(nb, b0 + per);
  auto gsize = [&](int b) { return group_size(a, b < a.n4 ? MOE_POOL_FP4 : MOE_POOL_INT2); };
  int np = 0, ng = 0;
  for (int b = b0; b < b1; ++b) {
    np += cnt[b];
    ng += (cnt[b] + gsize(b) - 1) / gsize(b);
  }
  int V, ngroups;
  int pos = block_exclusive_scan(np, ws, &V);
  int gi = block_exclusive_scan(ng, ws, &ngroups);
  for (int b = b0; b < b1; ++b) {
    cur[b] = pos;
    const int gs = gsize(b);
    for (int j = 0; j < cnt[b]; j += gs) {
      Group g;
      g.pool = b < a.n4 ? MOE_POOL_FP4 : MOE_POOL_INT2;
      g.slot = b < a.n4 ? b : b - a.n4;
      g.begin = pos + j;
      g.count = min(gs, cnt[b] - j);
      a.groups[gi++] = g;
    }
    pos += cnt[b];
  }
  __syncthreads();
  if (warp == 0) {
    for (int c0 = 0; c0 < P; c0 += 32) {
      const int p = c0 + lane;
      const int b = p < P ? binv[p] : -1;
      const unsigned m = __match_any_sync(0xffffffffu, b);
      const int base = b >= 0 ? cur[b] : 0;
      __syncwarp();
      if (b >= 0) {
        a.perm[base + __popc(m & ((1u << lane) - 1u))] = p;
        if (lane == __ffs(m) - 1) cur[b] = base + __popc(m);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  if (tid == 0) plan_finish(a, ngroups, scal[0] != 0);
}

__global__ void __launch_bounds__(1024) plan_kernel(FwdArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  pdl_launch_dependents();  // the block-scaled GEMM sets itself up meanwhile
  pdl_wait();               // launched early behind the slot ensure
  if (blockIdx.x > 0 && a.xhi) {
    plan_mx8_rows(a, blockIdx.x - 1, reinterpret_cast<int*>(smem_raw + 256),
                  reinterpret_cast<unsigned long long*>(smem_raw + 1024));
    if (!a.tags) return;  // the fp16 copy below serves only the 2-bit pairs' CUDA-core kernels then
    __syncthreads();
  }
  if (blockIdx.x > 0) {
    // activation prep for token t
    float* red = reinterpret_cast<float*>(smem_raw);
    const int t = blockIdx.x - 1;
    const uint16_t* xr = a.x + (size_t)t * a.H;
    float amax = 0.f;
    for (int n = threadIdx.x; n < a.H; n += blockDim.x)
      amax = fmaxf(amax, fabsf(__uint_as_float((uint32_t)xr[n] << 16)));
    amax = block_max(amax, red);
    const int sg = pow2_exponent(amax);
    for (int n = threadIdx.x; n < a.H; n += blockDim.x)
      a.xs[(size_t)t * a.H + n] = __float2half_rn(ldexpf(__uint_as_float((uint32_t)xr[n] << 16), -sg));
    if (threadIdx.x == 0) a.xsig[t] = sg;
    return;
  }
  // block 0: group kept pairs by (pool, slot); a routed-GEMM pass has no GEMV
  // groups (its grouping kernels check the slots), only the activation prep
  if (a.routed_gemm) return;
  if (a.n4 + a.n2 <= kPlanBins) return plan_groups_counting(a, smem_raw);
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem_raw);
  int* ws = reinterpret_cast<int*>(keys + kMaxPlanPairs);
  int* scal = ws + 34;
  const int P = a.P;
  int NP = 1;
  while (NP < P) NP <<= 1;
  const int tid = threadIdx.x, NT = blockDim.x;
  if (tid == 0) scal[0] = 0;
  __syncthreads();
  for (int p = tid; p < NP; p += NT) {
    unsigned long long key = p < P ? plan_key(a, p) : ~0ull;
    if (key == ~0ull - 1) {
      scal[0] = 1;
      key = ~0ull;
    }
    keys[p] = key;
  }
  __syncthreads();
  for (int size = 2; size <= NP; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < NP / 2; i += NT) {
        const int pos = 2 * i - (i & (stride - 1));
        const int par = pos + stride;
        const bool up = (pos & size) == 0;
        const unsigned long long x = keys[pos], y = keys[par];
        if ((x > y) == up) {
          keys[pos] = y;
          keys[par] = x;
        }
      }
      __syncthreads();
    }
  }
  // groups: runs of equal (pool, slot), cut every kG pairs.  Run starts are
  // compacted in order; each pair finds its run by binary search.
  int* starts = scal + 4;  // [NP]
  const int per = (NP + NT - 1) / NT;
  const int i0 = min(NP, tid * per), i1 = min(NP, i0 + per);
  int ns = 0, nv = 0;
  for (int i = i0; i < i1; ++i) {
    const unsigned long long key = keys[i];
    if (key == ~0ull) break;
    ++nv;
    ns += (i == 0 || (keys[i - 1] >> 32) != (key >> 32));
  }
  int NS, V;
  int sb = block_exclusive_scan(ns, ws, &NS);
  block_exclusive_scan(nv, ws, &V);
  for (int i = i0; i < i1; ++i) {
    const unsigned long long key = keys[i];
    if (key == ~0ull) break;
    if (i == 0 || (keys[i - 1] >> 32) != (key >> 32)) starts[sb++] = i;
  }
  __syncthreads();
  auto run_of = [&](int i) {
    int lo = 0, hi = NS;  // last start <= i
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (starts[mid] <= i) lo = mid; else hi = mid;
    }
    return lo;
  };
  // runs of a pool the warp-MMA kernels take are cut every a.mma_group pairs
  auto gsize = [&](unsigned long long key) { return group_size(a, (int)(key >> 62)); };
  int ng = 0;
  for (int i = i0; i < min(i1, V); ++i) ng += ((i - starts[run_of(i)]) % gsize(keys[i])) == 0;
  int ngroups;
  int gi = block_exclusive_scan(ng, ws, &ngroups);
  for (int i = i0; i < min(i1, V); ++i) {
    const unsigned long long key = keys[i];
    a.perm[i] = (int)(key & 0xffffffffu);
    const int r = run_of(i);
    const int gs = gsize(key);
    if ((i - starts[r]) % gs) continue;
    const int run_end = r + 1 < NS ? starts[r + 1] : V;
    Group g;
    g.pool = (int)(key >> 62);
    g.slot = (int)((key >> 32) & 0x3fffffffu);
    g.begin = i;
    g.count = min(gs, run_end - i);
    a.groups[gi++] = g;
  }
  __syncthreads();
  if (tid == 0) plan_finish(a, ngroups, scal[0] != 0);
}

// ---------------------------------------------------------- gate/up kernel --

// A work item's group is checked against the buffers it indexes before any
// access; a bad group (which the plan never produces) is skipped and flagged.
__device__ __forceinline__ bool group_ok(const FwdArgs& a, const Group& g) {
  if (g.pool < 0 || g.pool > 2 || g.count < 1 || g.count > group_size(a, g.pool)) return false;
  if (g.pool == MOE_POOL_SHARED) return a.shared != nullptr && g.begin >= 0 && g.begin + g.count <= a.T;
  const int npool = g.pool == MOE_POOL_FP4 ? a.n4 : (g.pool == MOE_POOL_INT2 ? a.n2 : 0);
  return g.slot >= 0 && g.slot < npool && g.begin >= 0 && g.begin + g.count <= a.P;
}

__device__ __forceinline__ int n_groups_checked(const FwdArgs& a) {
  const int n = a.hdr[0];
  const int cap = a.P + (a.T + kG - 1) / kG + 1;
  return (n < 0 || n > cap) ? 0 : n;
}

__device__ __forceinline__ const uint8_t* expert_base(const FwdArgs& a, int pool, int slot) {
  if (pool == MOE_POOL_FP4) return a.fp4 + (size_t)slot * a.b4;
  if (pool == MOE_POOL_INT2) return a.int2 + (size_t)slot * a.b2;
  return a.shared;
}


// ------------------------------------------------- two-deep row pipelining --
// For FP4 groups of one or two tokens the per-row compute is short, so a warp
// loads the codes of its next row pair before it computes the current one:
// twice the bytes in flight per warp.
template <int CPL>
struct Fp4Rows {
  uint4 q0[CPL], q1[CPL];
  uint32_t e0[CPL], e1[CPL];
};

template <int CPL>
__device__ __forceinline__ void fp4_load(Fp4Rows<CPL>& b, const uint8_t* c0, const uint8_t* s0, const uint8_t* c1,
                                         const uint8_t* s1) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const int c = lane + 32 * i;
    b.q0[i] = ld_stream_v4(c0 + (size_t)c * 16);
    b.q1[i] = ld_stream_v4(c1 + (size_t)c * 16);
    b.e0[i] = __ldg(s0 + c);
    b.e1[i] = __ldg(s1 + c);
  }
}

template <int CPL, int NT>
__device__ __forceinline__ void fp4_compute(const Fp4Rows<CPL>& b, const uint4* xs, int xstride, float* a0,
                                            float* a1) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < NT; ++t) a0[t] = a1[t] = 0.f;
#pragma unroll
  for (int i = 0; i < CPL; ++i) chunk_fp4<NT>(b.q0[i], b.e0[i], b.q1[i], b.e1[i], lane + 32 * i, xs, xstride, NT, a0, a1);
}

// Rows of one gate/up work item for a group of exactly NT tokens.
template <int KH, int NT>
__device__ __forceinline__ void gateup_rows(const FwdArgs& a, const Group& g, int tile, const uint4* xs,
                                            const int* tok, const int* hrow, int H, int I) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint8_t* ex = expert_base(a, g.pool, g.slot);
  const MatView w1 = mat_view(g.pool, ex, H, I, 0);
  const MatView w3 = mat_view(g.pool, ex, H, I, 1);
  if constexpr (KH > 0 && KH <= 2048 && KH % 1024 == 0 && NT <= 2) {
    if (g.pool == MOE_POOL_FP4 && I % kRowsGateUp == 0) {
      constexpr int CPL = KH / 1024;
      constexpr int NR = kRowsGateUp / (kFwdThreads / 32);  // row pairs per warp
      Fp4Rows<CPL> buf[2];
      auto load = [&](int j, Fp4Rows<CPL>& b) {
        const int n = tile * kRowsGateUp + warp + j * (kFwdThreads / 32);
        fp4_load<CPL>(b, w1.codes + (size_t)n * (H / 2), w1.scales + (size_t)n * (H / 32),
                      w3.codes + (size_t)n * (H / 2), w3.scales + (size_t)n * (H / 32));
      };
      load(0, buf[0]);
#pragma unroll
      for (int j = 0; j < NR; ++j) {
        if (j + 1 < NR) load(j + 1, buf[(j + 1) & 1]);
        float ag[NT], au[NT];
        fp4_compute<CPL, NT>(buf[j & 1], xs, H / 8, ag, au);
        warp_allreduce<NT>(ag);
        warp_allreduce<NT>(au);
        const int n = tile * kRowsGateUp + warp + j * (kFwdThreads / 32);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (t == lane) {
            const int sg = a.xsig[tok[t]];
            const float gv = ldexpf(ag[t], sg);
            const float uv = ldexpf(au[t], sg);
            a.h[(size_t)hrow[t] * I + n] = gv / (1.f + expf(-gv)) * uv;
          }
        }
      }
      return;
    }
  }
  for (int r = warp; r < kRowsGateUp; r += kFwdThreads / 32) {
    const int n = tile * kRowsGateUp + r;
    if (n >= I) break;
    float ag[NT], au[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) ag[t] = au[t] = 0.f;
    float rg = 1.f, ru = 1.f;
    if (g.pool == MOE_POOL_FP4) {
      rows_fp4<KH, NT>(w1.codes + (size_t)n * (H / 2), w1.scales + (size_t)n * (H / 32),
                       w3.codes + (size_t)n * (H / 2), w3.scales + (size_t)n * (H / 32), H, xs, NT, ag, au);
    } else if (g.pool == MOE_POOL_INT2) {
      rows_int2<KH, NT>(w1.codes + (size_t)n * (H / 4), w1.scales + (size_t)n * (H / 32),
                        w3.codes + (size_t)n * (H / 4), w3.scales + (size_t)n * (H / 32), H, xs, NT, ag, au);
    } else {
      rows_fp8<KH, NT>(w1.codes + (size_t)n * H, w3.codes + (size_t)n * H, H, xs, NT, ag, au);
      rg = __ldg(reinterpret_cast<const float*>(w1.scales) + n);
      ru = __ldg(reinterpret_cast<const float*>(w3.scales) + n);
    }
    warp_allreduce<NT>(ag);
    warp_allreduce<NT>(au);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t == lane) {
        const int sg = a.xsig[tok[t]];
        const float gv = ldexpf(ag[t] * rg, sg);
        const float uv = ldexpf(au[t] * ru, sg);
        a.h[(size_t)hrow[t] * I + n] = gv / (1.f + expf(-gv)) * uv;
      }
    }
  }
}

// Items (group, tile) are taken with a grid stride, so the token groups of one
// popular expert run at about the same time and its re-read rows hit L2; a
// group's activations are restaged only when the group changes.
template <int KH>
__global__ void __launch_bounds__(kFwdThreads, 2) gateup_kernel(FwdArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint4* xs = reinterpret_cast<uint4*>(smem_raw);
  int* tok = reinterpret_cast<int*>(smem_raw + (size_t)kG * a.H * 2);
  int* hrow = tok + kG;
  const int H = KH > 0 ? KH : a.H;
  const int I = a.I;
  const int tiles = (I + kRowsGateUp - 1) / kRowsGateUp;
  const long long n_items = (long long)n_groups_checked(a) * tiles;
  int staged = -1;
  for (long long item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int gi = (int)(item / tiles);
    const int tile = (int)(item % tiles);
    const Group g = a.groups[gi];
    if (g.pool >= 0 && g.pool < 31 && ((a.gemv_skip >> g.pool) & 1)) continue;
    if (!group_ok(a, g)) {
      if (threadIdx.x == 0 && a.err) *a.err = MOE_ERR_INVALID;
      continue;
    }
    if (gi != staged) {
      __syncthreads();  // the previous group's rows are done with xs
      if (threadIdx.x < g.count) {
        const int i = threadIdx.x;
        if (g.pool == MOE_POOL_SHARED) {
          tok[i] = g.begin + i;
          hrow[i] = a.P + g.begin + i;
        } else {
          const int p = min(max(a.perm[g.begin + i], 0), a.P - 1);
          tok[i] = p / a.k;
          hrow[i] = p;
        }
      }
      __syncthreads();
      stage_rows(g.pool, H, g.count, [&](int i) { return a.xs + (size_t)tok[i] * H; }, xs);
      __syncthreads();
      staged = gi;
    }
    switch (g.count) {
      case 1: gateup_rows<KH, 1>(a, g, tile, xs, tok, hrow, H, I); break;
      case 2: gateup_rows<KH, 2>(a, g, tile, xs, tok, hrow, H, I); break;
      case 3: gateup_rows<KH, 3>(a, g, tile, xs, tok, hrow, H, I); break;
      case 4: gateup_rows<KH, 4>(a, g, tile, xs, tok, hrow, H, I); break;
      case 5: gateup_rows<KH, 5>(a, g, tile, xs, tok, hrow, H, I); break;
      case 6: gateup_rows<KH, 6>(a, g, tile, xs, tok, hrow, H, I); break;
      case 7: gateup_rows<KH, 7>(a, g, tile, xs, tok, hrow, H, I); break;
      default: gateup_rows<KH, 8>(a, g, tile, xs, tok, hrow, H, I); break;
    }
  }
}

// -------------------------------------------------------------- down kernel --

template <int KI, int NT>
__device__ __forceinline__ void down_rows(const FwdArgs& a, const Group& g, int tile, const uint4* xs,
                                          const int* hrow, const int* sig, int H, int I) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint8_t* ex = expert_base(a, g.pool, g.slot);
  const MatView w2 = mat_view(g.pool, ex, H, I, 2);
  if constexpr (KI > 0 && KI % 1024 == 0 && NT <= 2) {
    if (g.pool == MOE_POOL_FP4 && H % kRowsDown == 0) {
      constexpr int CPL = KI / 1024;
      constexpr int NR = kRowsDown / (2 * (kFwdThreads / 32));  // row pairs per warp
      Fp4Rows<CPL> buf[2];
      auto load = [&](int j, Fp4Rows<CPL>& b) {
        const int n = tile * kRowsDown + 2 * warp + j * 2 * (kFwdThreads / 32);
        fp4_load<CPL>(b, w2.codes + (size_t)n * (I / 2), w2.scales + (size_t)n * (I / 32),
                      w2.codes + (size_t)(n + 1) * (I / 2), w2.scales + (size_t)(n + 1) * (I / 32));
      };
      load(0, buf[0]);
#pragma unroll
      for (int j = 0; j < NR; ++j) {
        if (j + 1 < NR) load(j + 1, buf[(j + 1) & 1]);
        float a0[NT], a1[NT];
        fp4_compute<CPL, NT>(buf[j & 1], xs, I / 8, a0, a1);
        warp_allreduce<NT>(a0);
        warp_allreduce<NT>(a1);
        const int n = tile * kRowsDown + 2 * warp + j * 2 * (kFwdThreads / 32);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (lane == t) a.o[(size_t)hrow[t] * H + n] = ldexpf(a0[t], sig[t]);
          if (lane == 16 + t) a.o[(size_t)hrow[t] * H + n + 1] = ldexpf(a1[t], sig[t]);
        }
      }
      return;
    }
  }
  for (int r = 2 * warp; r < kRowsDown; r += 2 * (kFwdThreads / 32)) {
    const int n = tile * kRowsDown + r;
    if (n >= H) break;
    const int n1 = min(n + 1, H - 1);
    float a0[NT], a1[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) a0[t] = a1[t] = 0.f;
    float r0 = 1.f, r1 = 1.f;
    if (g.pool == MOE_POOL_FP4) {
      rows_fp4<KI, NT>(w2.codes + (size_t)n * (I / 2), w2.scales + (size_t)n * (I / 32),
                       w2.codes + (size_t)n1 * (I / 2), w2.scales + (size_t)n1 * (I / 32), I, xs, NT, a0, a1);
    } else if (g.pool == MOE_POOL_INT2) {
      rows_int2<KI, NT>(w2.codes + (size_t)n * (I / 4), w2.scales + (size_t)n * (I / 32),
                        w2.codes + (size_t)n1 * (I / 4), w2.scales + (size_t)n1 * (I / 32), I, xs, NT, a0, a1);
    } else {
      rows_fp8<KI, NT>(w2.codes + (size_t)n * I, w2.codes + (size_t)n1 * I, I, xs, NT, a0, a1);
      r0 = __ldg(reinterpret_cast<const float*>(w2.scales) + n);
      r1 = __ldg(reinterpret_cast<const float*>(w2.scales) + n1);
    }
    warp_allreduce<NT>(a0);
    warp_allreduce<NT>(a1);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (lane == t) a.o[(size_t)hrow[t] * H + n] = ldexpf(a0[t] * r0, sig[t]);
      if (lane == 16 + t && n + 1 < H) a.o[(size_t)hrow[t] * H + n + 1] = ldexpf(a1[t] * r1, sig[t]);
    }
  }
}

template <int KI>
__global__ void __launch_bounds__(kFwdThreads, 2) down_kernel(FwdArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int H = a.H;
  const int I = KI > 0 ? KI : a.I;
  uint4* xs = reinterpret_cast<uint4*>(smem_raw);
  __half* hh = reinterpret_cast<__half*>(smem_raw + (size_t)kG * I * 2);  // [kG][I] natural order
  int* hrow = reinterpret_cast<int*>(smem_raw + (size_t)kG * I * 4);
  int* sig = hrow + kG;
  const int tiles = (H + kRowsDown - 1) / kRowsDown;
  const long long n_items = (long long)n_groups_checked(a) * tiles;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int staged = -1;
  for (long long item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int gi = (int)(item / tiles);
    const int tile = (int)(item % tiles);
    const Group g = a.groups[gi];
    if (g.pool >= 0 && g.pool < 31 && ((a.gemv_skip >> g.pool) & 1)) continue;
    if (!group_ok(a, g)) {
      if (threadIdx.x == 0 && a.err) *a.err = MOE_ERR_INVALID;
      continue;
    }
    if (gi != staged) {
      __syncthreads();
      if (threadIdx.x < g.count) {
        const int i = threadIdx.x;
        const int p = g.pool == MOE_POOL_SHARED ? 0 : a.perm[g.begin + i];
        hrow[i] = g.pool == MOE_POOL_SHARED ? a.P + g.begin + i : min(max(p, 0), a.P - 1);
      }
      __syncthreads();
      // per-row power-of-two scale of h, then fp16 rows in natural order
      for (int i = warp; i < g.count; i += kFwdThreads / 32) {
        const float* src = a.h + (size_t)hrow[i] * I;
        float m = 0.f;
        for (int n = lane; n < I; n += 32) m = fmaxf(m, fabsf(src[n]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const int sg = pow2_exponent(m);
        if (lane == 0) sig[i] = sg;
        for (int n = lane; n < I; n += 32) hh[(size_t)i * I + n] = __float2half_rn(ldexpf(src[n], -sg));
      }
      __syncthreads();
      stage_rows(g.pool, I, g.count, [&](int i) { return (const __half*)(hh + (size_t)i * I); }, xs);
      __syncthreads();
      staged = gi;
    }
    switch (g.count) {
      case 1: down_rows<KI, 1>(a, g, tile, xs, hrow, sig, H, I); break;
      case 2: down_rows<KI, 2>(a, g, tile, xs, hrow, sig, H, I); break;
      case 3: down_rows<KI, 3>(a, g, tile, xs, hrow, sig, H, I); break;
      case 4: down_rows<KI, 4>(a, g, tile, xs, hrow, sig, H, I); break;
      case 5: down_rows<KI, 5>(a, g, tile, xs, hrow, sig, H, I); break;
      case 6: down_rows<KI, 6>(a, g, tile, xs, hrow, sig, H, I); break;
      case 7: down_rows<KI, 7>(a, g, tile, xs, hrow, sig, H, I); break;
      default: down_rows<KI, 8>(a, g, tile, xs, hrow, sig, H, I); break;
    }
  }
}

}  // namespace moe

#include "decode_mma.cuh"

namespace moe {

// ------------------------------------------------------------ combine kernel --

// Four consecutive outputs per thread (16-byte loads of o, all k issued before
// use); per element the same fmaf chain in rank order as one element at a time.
__global__ void __launch_bounds__(256) combine_kernel(FwdArgs a) {
  pdl_wait();  // launched early behind the block-scaled down GEMM
  const int t = blockIdx.y;
  __shared__ float wk[64];
  __shared__ int pk[64];
  if (threadIdx.x < a.k) {
    const int p = t * a.k + threadIdx.x;
    const int sl = a.slots[p];
    const int tag = a.tags ? (int)a.tags[p] : MOE_TAG_FP4;
    const int npool = tag == MOE_TAG_INT2 ? a.n2 : a.n4;
    const bool keep = sl >= 0 && (tag == MOE_TAG_FP4 || tag == MOE_TAG_INT2) && sl < npool;
    wk[threadIdx.x] = keep ? a.w[p] : 0.f;
    pk[threadIdx.x] = keep ? p : -1;
  }
  __syncthreads();
  for (int n = 4 * (blockIdx.x * blockDim.x + threadIdx.x); n < a.H; n += 4 * gridDim.x * blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int j = 0; j < a.k; ++j) {
      if (pk[j] < 0) continue;
      const float4 v = *reinterpret_cast<const float4*>(a.o + (size_t)pk[j] * a.H + n);
      const float wj = wk[j];
      acc.x = fmaf(wj, v.x, acc.x);
      acc.y = fmaf(wj, v.y, acc.y);
      acc.z = fmaf(wj, v.z, acc.z);
      acc.w = fmaf(wj, v.w, acc.w);
    }
    if (a.shared) {
      const float4 v = *reinterpret_cast<const float4*>(a.o + (size_t)(a.P + t) * a.H + n);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    uint2 out;
    out.x = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.x)) |
            ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.y)) << 16);
    out.y = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.z)) |
            ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.w)) << 16);
    uint16_t* dst = a.y + (size_t)t * a.H + n;
    if (((uintptr_t)dst & 7) == 0) {
      *reinterpret_cast<uint2*>(dst) = out;
    } else {  // a caller's y need only be 2-byte aligned
      dst[0] = (uint16_t)out.x;
      dst[1] = (uint16_t)(out.x >> 16);
      dst[2] = (uint16_t)out.y;
      dst[3] = (uint16_t)(out.y >> 16);
    }
  }
}

// --------------------------------------------------------- dequant debug --

__global__ void dequant_kernel(const uint8_t* expert, int pool, int H, int I, int m, float* out) {
  const MatView v = mat_view(pool, expert, H, I, m);
  const size_t total = (size_t)v.N * v.K;
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx * 16 < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    // 16 consecutive weights of one row
    const size_t e0 = idx * 16;
    const int n = (int)(e0 / v.K), kk = (int)(e0 % v.K);
    float* o = out + e0;
    if (pool == MOE_POOL_FP4) {
      const uint8_t* c = v.codes + (size_t)n * (v.K / 2) + kk / 2;
      const float s = e8m0_f32(v.scales[(size_t)n * (v.K / 32) + kk / 32]);
      __half2 w[8];
      fp4_word_to_h2(*reinterpret_cast<const uint32_t*>(c), w);
      fp4_word_to_h2(*reinterpret_cast<const uint32_t*>(c + 4), w + 4);
      for (int i = 0; i < 8; ++i) {
        const float2 f = __half22float2(w[i]);
        o[2 * i] = f.x * s;
        o[2 * i + 1] = f.y * s;
      }
    } else if (pool == MOE_POOL_INT2) {
      const uint8_t* c = v.codes + (size_t)n * (v.K / 4) + kk / 4;
      const uint8_t sb = v.scales[(size_t)n * (v.K / 32) + kk / 32];
      const float s = __half22float2(e4m3x2_to_h2(sb)).x;
      __half2 w[8];
      int2_word_to_h2(*reinterpret_cast<const uint32_t*>(c), w);
      for (int i = 0; i < 8; ++i) {
        const float2 f = __half22float2(w[i]);
        o[i] = f.x * s;
        o[i + 8] = f.y * s;
      }
    } else {
      const uint8_t* c = v.codes + (size_t)n * v.K + kk;
      const float s = reinterpret_cast<const float*>(v.scales)[n];
      for (int i = 0; i < 8; ++i) {
        const uint32_t two = (uint32_t)c[2 * i] | ((uint32_t)c[2 * i + 1] << 8);
        const float2 f = __half22float2(e4m3x2_to_h2(two));
        o[2 * i] = f.x * s;
        o[2 * i + 1] = f.y * s;
      }
    }
  }
}

// -------------------------------------------------------------- rms carry --

__global__ void __launch_bounds__(256) rms_carry_kernel(const uint16_t* y, int H, float eps, uint16_t* xn) {
  __shared__ float red[33];
  const int t = blockIdx.x;
  const uint16_t* yr = y + (size_t)t * H;
  float ss = 0.f;
  for (int n = threadIdx.x; n < H; n += blockDim.x) {
    const float v = __uint_as_float((uint32_t)yr[n] << 16);
    ss = fmaf(v, v, ss);
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) red[wid] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += red[i];
    red[32] = 1.f / sqrtf(s / (float)H + eps);
  }
  __syncthreads();
  const float r = red[32];
  for (int n = threadIdx.x; n < H; n += blockDim.x)
    xn[(size_t)t * H + n] =
        __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float((uint32_t)yr[n] << 16) * r));
}

// ------------------------------------------------------------------- host --

// SM count of the current device.
static int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

template <typename K>
static moe_status set_smem(K kernel, size_t bytes) {
  if (bytes > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute((const void*)kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  }
  return MOE_OK;
}

template <typename K>
static int persistent_grid(K kernel, size_t smem, long long max_items) {
  int per_sm = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kFwdThreads, smem);
  if (per_sm < 1) per_sm = 1;
  long long g = (long long)sm_count() * per_sm;
  if (max_items < g) g = max_items;
  return (int)(g < 1 ? 1 : g);
}

template <typename K>
static int mma_grid(K kernel, size_t smem, long long max_items) {
  int per_sm = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kMmaThreads, smem);
  if (per_sm < 1) per_sm = 1;
  long long g = (long long)sm_count() * per_sm;
  if (max_items < g) g = max_items;
  return (int)(g < 1 ? 1 : g);
}

// Shapes the warp-MMA kernels take: K of every matrix a multiple of 256 (FP4
// steps of two 128-element chunks), whole gate/up and down tiles.
static bool mma_supported(const moe_expert_views* v) {
  return v->H % 512 == 0 && v->I % 512 == 0 && v->I % kMmaFeat == 0 && v->H % kMmaRowsDown == 0;
}

// Decode batches of at most this many tokens take the warp-MMA kernels for their
// FP4 and shared-expert groups (0: never); larger ones from kGemmMinPairs pairs
// take the tcgen05 grouped GEMM (moe_set_option).
static int g_mma_max_tokens = 64;
constexpr int kMmaMinTokens = 2;
// Of those, batches from this many tokens take the block-scaled tcgen05 GEMM
// (decode_mx8.cu) instead of the warp-MMA kernels (moe_set_option).
static int g_mx8_min_tokens = 2;

static moe_status validate_views(const moe_expert_views* v) {
  MOE_ARG(v != nullptr, "views is null");
  MOE_ARG(v->H > 0 && v->I > 0 && v->H % 32 == 0 && v->I % 32 == 0, "H and I must be positive multiples of 32");
  MOE_ARG(v->H % 64 == 0 && v->I % 64 == 0 || v->int2_slots == nullptr,
          "the 2-bit pool needs H and I multiples of 64");
  MOE_ARG(v->fp4_slots == nullptr || ((uintptr_t)v->fp4_slots & 15) == 0, "fp4_slots must be 16-byte aligned");
  MOE_ARG(v->int2_slots == nullptr || ((uintptr_t)v->int2_slots & 15) == 0, "int2_slots must be 16-byte aligned");
  MOE_ARG(v->shared == nullptr || ((uintptr_t)v->shared & 15) == 0, "shared must be 16-byte aligned");
  return MOE_OK;
}

}  // namespace moe

namespace moe {
size_t prefill_workspace(int H, int I, int T, int k, int S);
moe_status prefill_forward(const moe_expert_views* v, const uint16_t* x, int T, int k, const int32_t* slots,
                           const float* w, uint16_t* y, void* workspace, size_t ws_bytes, int32_t* d_error,
                           cudaStream_t stream, int prec_mode = MOE_PREC_W4A16);
}  // namespace moe

using namespace moe;

extern "C" size_t moe_expert_forward_workspace(const moe_expert_views* v, int T, int k) {
  if (!v || T < 0 || k < 1) return 0;
  if ((long long)T * k > kMaxPlanPairs) return prefill_workspace(v->H, v->I, T, k, v->fp4_num_slots);
  return fwd_layout(v, T, k).total;
}

namespace moe {

// Options of one pass of the decode forward over a subset of the pairs.
struct FwdPass {
  bool shared = true;            // include the shared expert
  bool combine = true;           // finish with the router-weighted combine into y
  uint8_t* gemm_bufs = nullptr;  // grouped GEMM activation / h copies (else aliased into o / h)
  DownParts down;                // waits before the down matrices are read (per part of the slots)
};

static moe_status forward_pass(const moe_expert_views* v, const uint16_t* x, int T, int k, const int32_t* slots,
                               const int8_t* tags, const float* w, uint16_t* y, uint8_t* base, const FwdLayout& L,
                               int32_t* d_error, cudaStream_t stream, const FwdPass& pass) {
  moe_status st;
  FwdArgs a;
  a.H = v->H;
  a.I = v->I;
  a.T = T;
  a.k = k;
  a.P = T * k;
  a.fp4 = v->fp4_slots;
  a.n4 = v->fp4_slots ? v->fp4_num_slots : 0;
  a.int2 = v->int2_slots;
  a.n2 = v->int2_slots ? v->int2_num_slots : 0;
  a.shared = pass.shared ? v->shared : nullptr;
  a.b4 = fp4_bytes(v->H, v->I);
  a.b2 = int2_bytes(v->H, v->I);
  a.x = x;
  a.slots = slots;
  a.tags = tags;
  a.w = w;
  a.y = y;
  a.err = d_error;
  a.routed_gemm = L.gemm && tags == nullptr && d_error != nullptr && T > g_mma_max_tokens;
  // the warp-MMA kernels take the FP4 and shared-expert groups of decode batches
  // from two tokens on (a single token gives too few work items to fill the GPU;
  // the CUDA-core kernels keep more bytes in flight there)
  const bool mma = !a.routed_gemm && T >= kMmaMinTokens && T <= g_mma_max_tokens && mma_supported(v);
  a.gemv_skip = mma ? kMmaPoolMask : 0;
  // token tiles per group: one up to 8 tokens, else two (with four tiles per
  // group only two chunk buffers fit the registers, which measured slower)
  const int mma_nb = T <= 8 ? 1 : 2;
  // the block-scaled tcgen05 GEMM: groups of up to 64 tokens (one per expert
  // at these batch sizes); the plan reads x rows with 8-byte loads
  const bool mx8 = mma && L.mx8_ok && g_mx8_min_tokens > 0 && T >= g_mx8_min_tokens && ((uintptr_t)x & 7) == 0;
  a.mma_group = mma ? (mx8 ? kMx8MaxRows : 8 * mma_nb) : 0;
  Mx8Bufs mb{};
  if (mx8) mx8_carve(base + L.mx8, v->H, v->I, a.P + T, &mb);
  a.xhi = mx8 ? mb.xhi : nullptr;
  a.xlo = mx8 ? mb.xlo : nullptr;
  a.xsc = mx8 ? mb.xsc : nullptr;
  a.hdr = (int*)(base + L.hdr);
  a.perm = (int*)(base + L.perm);
  a.groups = (Group*)(base + L.groups);
  a.xsig = (int*)(base + L.xsig);
  a.xs = (__half*)(base + L.xs);
  a.h = (float*)(base + L.h);
  a.o = (float*)(base + L.o);
  a.hs16 = (__half*)(base + L.hs16);
  a.hsig = (int*)(base + L.hsig);

  if (a.routed_gemm) {
    // the gather reads x rows with 16-byte loads
    MOE_ARG(((uintptr_t)x & 15) == 0, "x must be 16-byte aligned for the grouped-GEMM path (T * k >= %d)",
            kGemmMinPairs);
    // FP4 routed pairs on the tensor cores; its 16-bit buffers (two activation
    // copies of P x H each, h of P x I) reuse the routed rows of the fp32 o and
    // h buffers, which the CUDA-core kernels do not touch in this mode, unless
    // the pass brings its own (a second pass must not overwrite the first
    // pass's outputs in o)
    GgBufs gb;
    gg_carve_index(base + L.gg, T, k, v->fp4_num_slots, &gb);
    const size_t P = (size_t)T * k;
    if (pass.gemm_bufs) {
      gb.xg = (uint16_t*)pass.gemm_bufs;
      gb.xg16 = (__half*)(pass.gemm_bufs + P * v->H * 2);
      gb.hs = (__nv_bfloat16*)(pass.gemm_bufs + P * v->H * 4);
    } else {
      gb.xg = (uint16_t*)a.o;
      gb.xg16 = (__half*)((uint8_t*)a.o + P * v->H * 2);
      gb.hs = (__nv_bfloat16*)a.h;
    }
    gb.o = a.o;
    if ((st = grouped_gemm_fp4(v, x, T, k, slots, gb, d_error, stream, pass.down)) != MOE_OK) return st;
  }
  // the plan groups the pairs and prepares the fp16 activations for the GEMV
  // kernels; a routed-GEMM pass without the shared expert runs none of them
  // (the grouping kernels of the GEMM check the slots)
  // the shared expert takes the tensor cores too when the routed pairs do
  const bool shared_gemm = a.routed_gemm && a.shared != nullptr;
  const bool gemv = !a.routed_gemm;
  if (gemv || shared_gemm) {
    const size_t plan_smem = std::max((size_t)kMaxPlanPairs * 12 + 64 * 4,
                                      (size_t)(2 * kPlanBins + kMaxPlanPairs + 64) * 4);
    if ((st = set_smem(plan_kernel, plan_smem)) != MOE_OK) return st;
    {
      ProfScope ps(MOE_K_PLAN, stream);
      cudaError_t le = launch_pdl(plan_kernel, dim3(1 + T), dim3(1024), plan_smem, stream, a);
      if (le != cudaSuccess) return cuda_fail(le, "plan_kernel");
    }
    if ((st = check_launch("plan_kernel")) != MOE_OK) return st;
  }
  if (shared_gemm) {
    // SwiGLU scratch in the shared expert's rows of h; output rows P .. P + T - 1 of o
    __nv_bfloat16* hs_sh = reinterpret_cast<__nv_bfloat16*>(a.h + (size_t)a.P * a.I);
    if ((st = grouped_gemm_shared_fp8(v, a.xs, a.xsig, T, hs_sh, a.o, a.P, d_error, stream)) != MOE_OK) return st;
  }

  const long long max_groups = (long long)T * k + (T + kG - 1) / kG + 1;
  if (mx8) {
    ProfScope ps(MOE_K_GATEUP, stream);
    if ((st = mx8_gemm(v, 0, T, k, a.shared != nullptr, (int)max_groups, a.P + T, a.hdr, a.groups, a.perm, mb,
                       a.o, d_error, stream)) != MOE_OK)
      return st;
  } else if (mma) {
    auto launch = [&](auto kernel) -> moe_status {
      moe_status s2 = set_smem(kernel, kMmaSmem);
      if (s2 != MOE_OK) return s2;
      ProfScope ps(MOE_K_GATEUP, stream);
      kernel<<<mma_grid(kernel, kMmaSmem, max_groups * (v->I / kMmaFeat)), kMmaThreads, kMmaSmem, stream>>>(a);
      return MOE_OK;
    };
    st = mma_nb == 1 ? launch(mma_gateup_kernel<1>) : launch(mma_gateup_kernel<2>);
    if (st != MOE_OK) return st;
  }
  if ((st = check_launch("mma_gateup_kernel")) != MOE_OK) return st;
  // the CUDA-core kernels: every group, or only the 2-bit ones beside the MMA kernels
  const bool gemv_run = gemv && (!mma || tags != nullptr);
  const size_t gu_smem = (size_t)kG * v->H * 2 + 2 * kG * 4;
  const long long gu_items = max_groups * ((v->I + kRowsGateUp - 1) / kRowsGateUp);
  if (!gemv_run) {
  } else if (v->H == 4096) {
    if ((st = set_smem(gateup_kernel<4096>, gu_smem)) != MOE_OK) return st;
    ProfScope ps(MOE_K_GATEUP, stream);
    gateup_kernel<4096><<<persistent_grid(gateup_kernel<4096>, gu_smem, gu_items), kFwdThreads, gu_smem, stream>>>(a);
  } else {
    if ((st = set_smem(gateup_kernel<0>, gu_smem)) != MOE_OK) return st;
    ProfScope ps(MOE_K_GATEUP, stream);
    gateup_kernel<0><<<persistent_grid(gateup_kernel<0>, gu_smem, gu_items), kFwdThreads, gu_smem, stream>>>(a);
  }
  if ((st = check_launch("gateup_kernel")) != MOE_OK) return st;

  // the down kernels read every slot's matrices: they wait for the last part
  if (gemv && pass.down.n >= 1 && pass.down.ready && pass.down.ready[pass.down.n - 1])
    MOE_CUDA(cudaStreamWaitEvent(stream, pass.down.ready[pass.down.n - 1], 0));
  if (mx8) {
    ProfScope ps(MOE_K_DOWN, stream);
    if ((st = mx8_gemm(v, 1, T, k, a.shared != nullptr, (int)max_groups, a.P + T, a.hdr, a.groups, a.perm, mb,
                       a.o, d_error, stream)) != MOE_OK)
      return st;
  } else if (mma) {
    {
      // h rows in fp16 with a power-of-two scale each (routed pairs and shared rows)
      const int rows = a.P + (a.shared ? T : 0);
      ProfScope ps(MOE_K_DOWN, stream);
      mma_hprep_kernel<<<std::min((rows + 7) / 8, sm_count() * 8), 256, 0, stream>>>(a.h, rows, a.I, a.hs16,
                                                                                      a.hsig);
    }
    if ((st = check_launch("mma_hprep_kernel")) != MOE_OK) return st;
    auto launch = [&](auto kernel) -> moe_status {
      moe_status s2 = set_smem(kernel, kMmaSmem);
      if (s2 != MOE_OK) return s2;
      ProfScope ps(MOE_K_DOWN, stream);
      kernel<<<mma_grid(kernel, kMmaSmem, max_groups * (v->H / kMmaRowsDown)), kMmaThreads, kMmaSmem, stream>>>(a);
      return MOE_OK;
    };
    st = mma_nb == 1 ? launch(mma_down_kernel<1>) : launch(mma_down_kernel<2>);
    if (st != MOE_OK) return st;
  }
  if ((st = check_launch("mma_down_kernel")) != MOE_OK) return st;
  const size_t dn_smem = (size_t)kG * v->I * 4 + 2 * kG * 4;
  const long long dn_items = max_groups * ((v->H + kRowsDown - 1) / kRowsDown);
  if (!gemv_run) {
  } else if (v->I == 2048) {
    if ((st = set_smem(down_kernel<2048>, dn_smem)) != MOE_OK) return st;
    ProfScope ps(MOE_K_DOWN, stream);
    down_kernel<2048><<<persistent_grid(down_kernel<2048>, dn_smem, dn_items), kFwdThreads, dn_smem, stream>>>(a);
  } else {
    if ((st = set_smem(down_kernel<0>, dn_smem)) != MOE_OK) return st;
    ProfScope ps(MOE_K_DOWN, stream);
    down_kernel<0><<<persistent_grid(down_kernel<0>, dn_smem, dn_items), kFwdThreads, dn_smem, stream>>>(a);
  }
  if ((st = check_launch("down_kernel")) != MOE_OK) return st;
  if (!pass.combine) return MOE_OK;

  dim3 cg((v->H / 4 + 255) / 256, T);
  ProfScope ps(MOE_K_COMBINE, stream);
  if (mx8) {
    cudaError_t le = launch_pdl(combine_kernel, cg, dim3(256), 0, stream, a);
    if (le != cudaSuccess) return cuda_fail(le, "combine_kernel");
  } else {
    combine_kernel<<<cg, 256, 0, stream>>>(a);
  }
  return check_launch("combine_kernel");
}

// Splits the pairs of a chunk by whether their slot is on the miss list, and
// the missed ones by the part of the list (as the part-wise copy divides it:
// part q holds entries [n * q / parts, n * (q + 1) / parts)): hit[p] keeps the
// slot of pairs whose expert was resident, miss[q * P + p] the slot of pairs
// whose expert is copied in with part q (every other entry -1).
__global__ void __launch_bounds__(1024) split_miss_kernel(const int32_t* slots, int P, const int32_t* miss_slot,
                                                          const int32_t* miss_count, int max_miss, int S,
                                                          int parts, int32_t* hit, int32_t* miss,
                                                          int slot_parts, int8_t* slot_part) {
  extern __shared__ int8_t part_of[];  // [S]: part of the slot's miss, -1 if not missed
  for (int i = threadIdx.x; i < S; i += blockDim.x) part_of[i] = -1;
  __syncthreads();
  const int n = min(max(*miss_count, 0), max_miss);
  const int np = parts > 1 ? parts : slot_parts;  // the partition the arrays or the slot index follow
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int sl = miss_slot[i];
    int q = 0;
    while (q + 1 < np && (long long)n * (q + 1) / np <= i) ++q;
    if (sl >= 0 && sl < S) part_of[sl] = (int8_t)q;
  }
  __syncthreads();
  if (slot_part && blockIdx.x == 0)
    for (int i = threadIdx.x; i < S; i += blockDim.x) slot_part[i] = part_of[i];
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < P; p += gridDim.x * blockDim.x) {
    const int sl = slots[p];
    const int q = (sl >= 0 && sl < S) ? part_of[sl] : -1;
    hit[p] = q >= 0 ? -1 : sl;
    if (parts > 1) {
      for (int r = 0; r < parts; ++r) miss[(size_t)r * P + p] = q == r ? sl : -1;
    } else {
      miss[p] = q >= 0 ? sl : -1;
    }
  }
}

static size_t overlap_extra(const moe_expert_views* v, int T, int k, const FwdLayout& L) {
  const size_t P = (size_t)T * k;
  size_t b = align256(P * 4) + align256((size_t)MOE_MAX_COPY_PARTS * P * 4) + align256((size_t)v->fp4_num_slots);
  if (L.gemm) b += align256(P * v->H * 4 + P * v->I * 2);
  return b;
}

}  // namespace moe

extern "C" moe_status moe_expert_forward(const moe_expert_views* v, const uint16_t* x, int T, int k,
                                         const int32_t* slots, const int8_t* tags, const float* w,
                                         uint16_t* y, void* workspace, size_t workspace_bytes,
                                         int32_t* d_error, cudaStream_t stream) {
  clear_error();
  moe_status st = validate_views(v);
  if (st != MOE_OK) return st;
  MOE_ARG(T >= 0 && k >= 1 && k <= 64, "need T >= 0 and 1 <= k <= 64");
  if (T == 0) return MOE_OK;
  MOE_ARG(x && slots && w && y && workspace, "null pointer");
  if ((long long)T * k > kMaxPlanPairs) {
    // prefill-sized batch: grouped GEMM on the tensor cores (FP4 pool only)
    MOE_ARG(tags == nullptr, "tags are not supported above %d pairs per call", kMaxPlanPairs);
    MOE_ARG(((uintptr_t)workspace & 255) == 0, "workspace must be 256-byte aligned");
    MOE_ARG(((uintptr_t)x & 15) == 0, "x must be 16-byte aligned");
    return prefill_forward(v, x, T, k, slots, w, y, workspace, workspace_bytes, d_error, stream);
  }
  MOE_ARG(((uintptr_t)workspace & 255) == 0, "workspace must be 256-byte aligned");
  const FwdLayout L = fwd_layout(v, T, k);
  MOE_ARG(workspace_bytes >= L.total, "workspace too small: %zu < %zu", workspace_bytes, L.total);
  MOE_ARG(v->fp4_slots || v->int2_slots, "no expert pool");
  if (d_error) MOE_CUDA(cudaMemsetAsync(d_error, 0, sizeof(int32_t), stream));
  return forward_pass(v, x, T, k, slots, tags, w, y, (uint8_t*)workspace, L, d_error, stream, FwdPass());
}

extern "C" size_t moe_expert_forward_overlap_workspace(const moe_expert_views* v, int T, int k) {
  if (!v || T < 0 || k < 1 || (long long)T * k > kMaxPlanPairs) return 0;
  const FwdLayout L = fwd_layout(v, T, k);
  return L.total + overlap_extra(v, T, k, L);
}

namespace moe {

// How the missed pairs follow their copies: `parts` passes over parts of the
// miss list, pass q after parts_done[q]; or (parts == 0, staged) one pass
// whose gate/up waits for gateup_ready and whose down work waits for
// down_ready[q] per part q of the slots (down_parts of them).
struct OverlapPlan {
  int parts = 1;
  const cudaEvent_t* parts_done = nullptr;
  cudaEvent_t gateup_ready = nullptr;
  int down_parts = 1;
  const cudaEvent_t* down_ready = nullptr;
};

static moe_status forward_overlap(const moe_expert_views* v, const uint16_t* x, int T, int k, const int32_t* slots,
                                  const float* w, const int32_t* d_miss_slot, const int32_t* d_miss_count,
                                  int max_miss, const OverlapPlan& plan, uint16_t* y, void* workspace,
                                  size_t workspace_bytes, int32_t* d_error, cudaStream_t stream) {
  moe_status st = validate_views(v);
  if (st != MOE_OK) return st;
  MOE_ARG(T >= 0 && k >= 1 && k <= 64, "need T >= 0 and 1 <= k <= 64");
  if (T == 0) return MOE_OK;
  MOE_ARG((long long)T * k <= kMaxPlanPairs, "T * k = %lld above the %d pairs of one overlapped call",
          (long long)T * k, kMaxPlanPairs);
  MOE_ARG(x && slots && w && y && workspace && d_miss_slot && d_miss_count, "null pointer");
  MOE_ARG(v->fp4_slots != nullptr, "no FP4 pool");
  MOE_ARG(max_miss >= 0, "max_miss < 0");
  MOE_ARG(((uintptr_t)workspace & 255) == 0, "workspace must be 256-byte aligned");
  const FwdLayout L = fwd_layout(v, T, k);
  const size_t need = L.total + overlap_extra(v, T, k, L);
  MOE_ARG(workspace_bytes >= need, "workspace too small: %zu < %zu", workspace_bytes, need);
  // workspace past the forward's own: hit slots [P], miss slots [parts][P],
  // the slots' part index [S], then the miss pass's GEMM buffers
  uint8_t* base = (uint8_t*)workspace;
  const size_t P = (size_t)T * k;
  const int S = v->fp4_num_slots;
  int32_t* hit = (int32_t*)(base + L.total);
  int32_t* miss = (int32_t*)(base + L.total + align256(P * 4));
  int8_t* slot_part = (int8_t*)(base + L.total + align256(P * 4) + align256((size_t)MOE_MAX_COPY_PARTS * P * 4));
  uint8_t* gemm_bufs = L.gemm ? (uint8_t*)slot_part + align256((size_t)S) : nullptr;
  const bool staged = plan.parts == 0;
  if (d_error) MOE_CUDA(cudaMemsetAsync(d_error, 0, sizeof(int32_t), stream));
  if ((st = set_smem(split_miss_kernel, (size_t)S)) != MOE_OK) return st;
  split_miss_kernel<<<(int)((P + 1023) / 1024), 1024, (size_t)S, stream>>>(
      slots, (int)P, d_miss_slot, d_miss_count, max_miss, S, staged ? 1 : plan.parts, hit, miss,
      staged ? plan.down_parts : 1, staged ? slot_part : nullptr);
  if ((st = check_launch("split_miss_kernel")) != MOE_OK) return st;
  // pass 1: pairs whose experts were resident, and the shared expert, while
  // the misses are still being copied
  FwdPass p1;
  p1.combine = false;
  if ((st = forward_pass(v, x, T, k, hit, nullptr, w, y, base, L, d_error, stream, p1)) != MOE_OK) return st;
  // then the missed pairs as their bytes land; the passes run in order on the
  // stream, so they can share the GEMM's buffers
  FwdPass p2;
  p2.shared = false;
  p2.combine = false;
  p2.gemm_bufs = gemm_bufs;
  if (staged) {
    // the gate/up matrices have landed: the first GEMM runs while the down
    // matrices are still on the way
    if (plan.gateup_ready) MOE_CUDA(cudaStreamWaitEvent(stream, plan.gateup_ready, 0));
    p2.down.n = plan.down_parts;
    p2.down.ready = plan.down_ready;
    p2.down.slot_part = slot_part;
    if ((st = forward_pass(v, x, T, k, miss, nullptr, w, y, base, L, d_error, stream, p2)) != MOE_OK) return st;
  } else {
    for (int q = 0; q < plan.parts; ++q) {
      if (plan.parts_done[q]) MOE_CUDA(cudaStreamWaitEvent(stream, plan.parts_done[q], 0));
      if ((st = forward_pass(v, x, T, k, miss + (size_t)q * P, nullptr, w, y, base, L, d_error, stream, p2)) !=
          MOE_OK)
        return st;
    }
  }
  // one combine over every pair of the chunk
  FwdArgs a{};
  a.H = v->H;
  a.I = v->I;
  a.T = T;
  a.k = k;
  a.P = (int)P;
  a.n4 = S;
  a.n2 = 0;
  a.shared = v->shared;
  a.slots = slots;
  a.tags = nullptr;
  a.w = w;
  a.y = y;
  a.o = (float*)(base + L.o);
  dim3 cg((v->H / 4 + 255) / 256, T);
  ProfScope ps(MOE_K_COMBINE, stream);
  combine_kernel<<<cg, 256, 0, stream>>>(a);
  return check_launch("combine_kernel");
}

}  // namespace moe

extern "C" moe_status moe_expert_forward_overlap_parts(const moe_expert_views* v, const uint16_t* x, int T, int k,
                                                       const int32_t* slots, const float* w,
                                                       const int32_t* d_miss_slot, const int32_t* d_miss_count,
                                                       int max_miss, int n_parts, const cudaEvent_t* parts_done,
                                                       uint16_t* y, void* workspace, size_t workspace_bytes,
                                                       int32_t* d_error, cudaStream_t stream) {
  clear_error();
  MOE_ARG(n_parts >= 1 && n_parts <= MOE_MAX_COPY_PARTS, "n_parts %d outside [1, %d]", n_parts,
          MOE_MAX_COPY_PARTS);
  MOE_ARG(parts_done != nullptr, "null pointer");
  OverlapPlan plan;
  plan.parts = n_parts;
  plan.parts_done = parts_done;
  return forward_overlap(v, x, T, k, slots, w, d_miss_slot, d_miss_count, max_miss, plan, y, workspace,
                         workspace_bytes, d_error, stream);
}

extern "C" moe_status moe_expert_forward_overlap_staged(const moe_expert_views* v, const uint16_t* x, int T, int k,
                                                        const int32_t* slots, const float* w,
                                                        const int32_t* d_miss_slot, const int32_t* d_miss_count,
                                                        int max_miss, cudaEvent_t gateup_ready, int n_down_parts,
                                                        const cudaEvent_t* down_ready, uint16_t* y,
                                                        void* workspace, size_t workspace_bytes, int32_t* d_error,
                                                        cudaStream_t stream) {
  clear_error();
  MOE_ARG(n_down_parts >= 1 && n_down_parts <= MOE_MAX_COPY_PARTS, "n_down_parts %d outside [1, %d]", n_down_parts,
          MOE_MAX_COPY_PARTS);
  MOE_ARG(down_ready != nullptr, "null pointer");
  OverlapPlan plan;
  plan.parts = 0;
  plan.gateup_ready = gateup_ready;
  plan.down_parts = n_down_parts;
  plan.down_ready = down_ready;
  return forward_overlap(v, x, T, k, slots, w, d_miss_slot, d_miss_count, max_miss, plan, y, workspace,
                         workspace_bytes, d_error, stream);
}

extern "C" moe_status moe_expert_forward_overlap(const moe_expert_views* v, const uint16_t* x, int T, int k,
                                                 const int32_t* slots, const float* w, const int32_t* d_miss_slot,
                                                 const int32_t* d_miss_count, int max_miss,
                                                 cudaEvent_t copies_done, uint16_t* y, void* workspace,
                                                 size_t workspace_bytes, int32_t* d_error, cudaStream_t stream) {
  return moe_expert_forward_overlap_parts(v, x, T, k, slots, w, d_miss_slot, d_miss_count, max_miss, 1,
                                          &copies_done, y, workspace, workspace_bytes, d_error, stream);
}

// ------------------------------------------------------ allocation-free entry --
// Scratch for moe_expert_forward_noalloc: a fixed array in device memory that
// every GPU loading this library holds until the process exits.  Host code
// cannot pass the array's name to a kernel (on the host it names a stand-in,
// not device memory), so its device address is looked up once per device.
constexpr size_t kNoAllocScratchBytes = (size_t)32 << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

static std::mutex g_noalloc_mu;
static void* g_noalloc_addr[128] = {};

static moe_status noalloc_scratch(void** out) {
  int dev = 0;
  MOE_CUDA(cudaGetDevice(&dev));
  MOE_ARG(dev >= 0 && dev < 128, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(fixed scratch)");
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return MOE_OK;
}

extern "C" moe_status moe_expert_forward_noalloc(const moe_expert_views* v, const uint16_t* x, int T, int k,
                                                 const int32_t* slots, const int8_t* tags, const float* w,
                                                 uint16_t* y, int32_t* d_error, cudaStream_t stream) {
  clear_error();
  moe_status st = validate_views(v);
  if (st != MOE_OK) return st;
  MOE_ARG(T >= 0 && k >= 1 && k <= 64, "need T >= 0 and 1 <= k <= 64");
  if (T == 0) return MOE_OK;
  MOE_ARG((long long)T * k <= kMaxPlanPairs, "T * k = %lld: the allocation-free call takes at most %d pairs",
          (long long)T * k, kMaxPlanPairs);
  const size_t need = fwd_layout(v, T, k).total;
  MOE_ARG(need <= kNoAllocScratchBytes,
          "this call needs %zu bytes of scratch but the fixed scratch holds %zu; pass fewer tokens per call", need,
          kNoAllocScratchBytes);
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != MOE_OK) return st;
  // nothing in the scratch has to start at zero: every region is written
  // by an earlier kernel of the same call before it is read
  return moe_expert_forward(v, x, T, k, slots, tags, w, y, scratch, kNoAllocScratchBytes, d_error, stream);
}

extern "C" moe_status moe_set_option(int option, int value, int* old_value) {
  clear_error();
  MOE_ARG(option == MOE_OPT_MMA_MAX_TOKENS || option == MOE_OPT_MX8_MIN_TOKENS, "unknown option %d", option);
  MOE_ARG(value >= 0, "option value must be >= 0");
  int& slot = option == MOE_OPT_MMA_MAX_TOKENS ? g_mma_max_tokens : g_mx8_min_tokens;
  if (old_value) *old_value = slot;
  slot = value;
  return MOE_OK;
}

extern "C" moe_status moe_dequant_debug(const moe_expert_views* v, int pool, int slot, int matrix,
                                        float* out, cudaStream_t stream) {
  clear_error();
  moe_status st = validate_views(v);
  if (st != MOE_OK) return st;
  MOE_ARG(out != nullptr, "out is null");
  MOE_ARG(matrix >= 0 && matrix <= 2, "matrix must be MOE_W1, MOE_W3 or MOE_W2");
  const uint8_t* ex = nullptr;
  if (pool == MOE_POOL_FP4) {
    MOE_ARG(v->fp4_slots && slot >= 0 && slot < v->fp4_num_slots, "bad FP4 slot");
    ex = v->fp4_slots + (size_t)slot * fp4_bytes(v->H, v->I);
  } else if (pool == MOE_POOL_INT2) {
    MOE_ARG(v->int2_slots && slot >= 0 && slot < v->int2_num_slots, "bad 2-bit slot");
    ex = v->int2_slots + (size_t)slot * int2_bytes(v->H, v->I);
  } else {
    MOE_ARG(pool == MOE_POOL_SHARED && v->shared, "bad pool");
    ex = v->shared;
  }
  const size_t n16 = (size_t)v->H * v->I / 16;
  const int blocks = (int)((n16 + 255) / 256 < 4096 ? (n16 + 255) / 256 : 4096);
  dequant_kernel<<<blocks, 256, 0, stream>>>(ex, pool, v->H, v->I, matrix, out);
  return check_launch("dequant_kernel");
}

extern "C" moe_status moe_rms_carry(const uint16_t* y, int T, int H, float eps, uint16_t* x_next,
                                    cudaStream_t stream) {
  clear_error();
  MOE_ARG(T >= 0 && H > 0, "bad sizes");
  if (T == 0) return MOE_OK;
  MOE_ARG(y && x_next, "null pointer");
  MOE_ARG(eps >= 0.f, "eps must be >= 0");
  ProfScope ps(MOE_K_CARRY, stream);
  rms_carry_kernel<<<T, 256, 0, stream>>>(y, H, eps, x_next);
  return check_launch("rms_carry_kernel");
}
