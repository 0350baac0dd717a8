// Grouped expert MLP for prefill-sized batches on the tcgen05 tensor cores.
//
// "Running DeepSeek-V4-Flash across four free GPUs", section "All four workers
// die, but only on prompts over 32 tokens": past T * top_k >= num_experts a
// prefill chunk touches most experts, and the expert work is one grouped GEMM
// over all tokens routed to each expert.  Weights are the MXFP4 experts of
// the slot pool (section "The model"); activations stay bf16 (W4A16, as every
// page runs its experts).
//
// Pipeline of one call:
//   group     pairs sorted by slot (stable counting sort, moe_group_pairs)
//   items     per slot, tiles of <= 256 rows of its pairs
//   gather    Xg[i] = x[token of the i-th sorted pair] (bf16 rows, 16-byte copies)
//   GEMM1     per (item, 128-feature tile): D0[128, n] = W1 . Xg^T and
//             D1[128, n] = W3 . Xg^T over K = H (same rows of both, so a
//             thread's TMEM lane holds gate and up of one feature); epilogue
//             h = SiLU(gate) * up -> bf16 rows of Hs
//   GEMM2     per (item, 128-feature tile): D[128, n] = W2 . Hs^T over K = I;
//             epilogue o[pair][feature] in fp32
//   combine   y_t = sum_j w_tj o_tj in rank order -> bf16
//
// GEMM CTA (512 threads): warp 12 lane 0 streams the raw FP4 codes of the A
// tiles by TMA into a staging ring, as far ahead as the ring allows; warp 14
// lane 0 loads the B tile by TMA straight into its 128-byte swizzled K-major
// layout, one stage per free operand slot; warps 0-11 decode the raw codes to
// 16-bit with the E8M0 scale folded in (exact) and store them in the same
// swizzled layout; warp 13 lane 0 issues tcgen05.mma.kind::f16 (M = 128,
// N = rows of the item rounded to 16, K = 16 per instruction) into two TMEM
// accumulators and commits each stage back to the producers; all 16 warps
// read TMEM with tcgen05.ld for the epilogue.  Every mbarrier wait gives up
// after one second and records MOE_ERR_TIMEOUT.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "grouped_gemm.cuh"
#include "tcgen05.cuh"
#include "mx.cuh"

namespace moe {

constexpr int kPfThreads = 512;   // 16 warps: 12 converters, raw producer, MMA, B producer, spare
constexpr int kPfMT = 2;          // 128-row weight tiles per CTA (two TMEM accumulators)
constexpr int kPfNMax = 256;      // rows per item (MMA N) of the item list
constexpr int kMxNMax = 224;      // rows per item of the block-scaled FP4 path (two 224-column accumulators)
constexpr int kPfKStep = 64;      // K elements per stage (128 bytes of bf16: one swizzle row)
constexpr int kPfBox = 64;        // rows per TMA box of the B operand
// Converter warps 0-11 form three groups of 128 threads; group g converts the
// K steps ks with ks % 3 == g, one A row per thread.  The converters' instruction
// stream bounds a K step, so three warps per scheduler keep more of it issuing.
constexpr int kPfConvGroups = 3;
constexpr int kPfConvThreads = 128;
constexpr int kPfConvWarps = kPfConvGroups * kPfConvThreads / 32;  // 12
constexpr int kWarpRaw = kPfConvWarps;       // raw FP4 code producer
constexpr int kWarpMma = kPfConvWarps + 1;   // TMEM allocation, MMA issue
constexpr int kWarpB = kPfConvWarps + 2;     // activation (B) producer
constexpr int kPfWarps = kPfThreads / 32;

// shared memory layout (offsets from a 1024-aligned base)
constexpr int kATile = 128 * 128;                 // 16 KB per 128-row tile
constexpr int kAStage = kPfMT * kATile;           // 32 KB
constexpr int kRawTile = kPfMT * 128 * 32;        // 8 KB of packed codes per stage

// Shapes of the GEMM CTA: items of up to 256 rows with three operand stages
// and a 4-deep raw-code ring (prefill: tensor-bound), or items of up to 64
// rows, whose smaller B stages leave room for four operand stages and an
// 8-deep ring (decode batches: a fourth stage lengthens the reuse distance of
// each A stage, which bounds a K step at small N; 64 KB of codes in flight per
// SM).  The FP8 shared expert keeps three stages and a 12-deep ring of 8 KB
// (six of its 16 KB stages).
template <int NMAX, int RAW, int STAGES>
struct PfCfg {
  static constexpr int kNMax = NMAX;
  static constexpr int kRaw = RAW;
  static constexpr int kStages = STAGES;  // A/B operand stages
  static constexpr int kBTile = NMAX * 128;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + STAGES * kAStage;
  static constexpr int kOffRaw = kOffB + STAGES * kBTile;
  static constexpr int kOffBar = kOffRaw + RAW * kRawTile;
  static constexpr int kSmem = kOffBar + 512 + 1024;  // barriers + alignment slack
  static_assert((2 * STAGES + 2 * RAW + 1) * 8 + 8 <= 512, "barrier area");
  static_assert(kSmem <= 232448, "shared memory per CTA");
};
using PfBig = PfCfg<256, 4, 3>;
using PfSmall = PfCfg<64, 8, 4>;
using PfShared = PfCfg<64, 12, 3>;  // FP8 shared expert: 16 KB raw stages, so a deeper ring

// kind::f16 instruction descriptor: D fp32, A and B both bf16 (or both fp16),
// both K-major, M = 128.
__device__ __forceinline__ uint32_t idesc_16bit(int n, bool bf16) {
  const uint32_t t = bf16 ? 1u : 0u;
  return (1u << 4) | (t << 7) | (t << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// One 64-wide K step of both accumulators, issued by one elected lane of a
// converged warp: four K = 16 MMAs per 128-row A tile (descriptor start
// addresses advance 32 bytes per slice inside the 128-byte swizzled rows),
// then a commit that arrives on `bar` once they complete.  `acc` = 0 starts
// the accumulators (first K step only).
__device__ __forceinline__ void mma_kstep_2x4(uint32_t d0, uint32_t d1, uint64_t a0, uint64_t a1, uint64_t b,
                                              uint32_t idesc, uint32_t acc, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred p, t, e;\n\t.reg .b64 a, bb;\n\t"
      "elect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %5, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %4, %6, p;\n\t"
      "add.s64 a, %2, 2;\n\tadd.s64 bb, %4, 2;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, bb, %6, t;\n\t"
      "add.s64 a, %2, 4;\n\tadd.s64 bb, %4, 4;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, bb, %6, t;\n\t"
      "add.s64 a, %2, 6;\n\tadd.s64 bb, %4, 6;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, bb, %6, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%1], %3, %4, %6, p;\n\t"
      "add.s64 a, %3, 2;\n\tadd.s64 bb, %4, 2;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%1], a, bb, %6, t;\n\t"
      "add.s64 a, %3, 4;\n\tadd.s64 bb, %4, 4;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%1], a, bb, %6, t;\n\t"
      "add.s64 a, %3, 6;\n\tadd.s64 bb, %4, 6;\n\t@e tcgen05.mma.cta_group::1.kind::f16 [%1], a, bb, %6, t;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%7];\n\t}" ::"r"(d0),
      "r"(d1), "l"(a0), "l"(a1), "l"(b), "r"(acc), "r"(idesc), "r"(su32(bar))
      : "memory");
}
// Eight E2M1 codes (one 32-bit word, element 2j in the low nibble of byte j)
// -> four 16-bit pairs times the block scale: the word is split into its four
// bytes by one mov, each byte converted by cvt.rn.f16x2.e2m1x2.
__device__ __forceinline__ void fp4x8_to_f16(uint32_t w, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(w));
}

// Four E4M3 codes (one 32-bit word, element j in byte j) -> two fp16 pairs (exact).
__device__ __forceinline__ void fp8x4_to_f16(uint32_t w, uint32_t& r0, uint32_t& r1) {
  asm("{\n\t.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, h0;\n\tcvt.rn.f16x2.e4m3x2 %1, h1;\n\t}"
      : "=r"(r0), "=r"(r1)
      : "r"(w));
}

// fp16 pair -> bf16 pair (exact for values with at most 8 significant bits)
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h) {
  uint32_t r;
  asm("{\n\t.reg .b16 l, u, bl, bu;\n\tmov.b32 {l, u}, %1;\n\tcvt.rn.bf16.f16 bl, l;\n\tcvt.rn.bf16.f16 bu, u;\n\t"
      "mov.b32 %0, {bl, bu};\n\t}"
      : "=r"(r)
      : "r"(h));
  return r;
}

// fp16 pair times the block scale 2^(e-127) given as fp16x2: exact when e is
// within [kF16ScaleLo, kF16ScaleHi].
__device__ __forceinline__ uint32_t hmul2_f16(uint32_t a, uint32_t s) {
  __half2 v = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<const __half2*>(&s));
  return *reinterpret_cast<uint32_t*>(&v);
}

// fp16 pair (exact E2M1 values) -> bf16 pair times the block scale: exact for
// every E8M0 scale.
__device__ __forceinline__ uint32_t f16x2_to_bf16x2_scaled(uint32_t h, uint32_t scale2) {
  uint32_t r;
  asm("{\n\t.reg .b16 l, u, bl, bu;\n\tmov.b32 {l, u}, %1;\n\tcvt.rn.bf16.f16 bl, l;\n\tcvt.rn.bf16.f16 bu, u;\n\t"
      "mov.b32 %0, {bl, bu};\n\t}"
      : "=r"(r)
      : "r"(h));
  __nv_bfloat162 v = __hmul2(*reinterpret_cast<__nv_bfloat162*>(&r), *reinterpret_cast<const __nv_bfloat162*>(&scale2));
  return *reinterpret_cast<uint32_t*>(&v);
}

// E8M0 range for which E2M1 x 2^(e-127) is a normal fp16 (or zero) with an
// fp16-normal scale: 2^-12 <= 0.5 * 2^(e-127) and 6 * 2^(e-127) <= 49152.
constexpr uint32_t kF16ScaleLo = 115, kF16ScaleHi = 140;

__device__ __forceinline__ uint32_t e8m0_f16x2(uint32_t e) {
  const uint32_t h = (e - 127 + 15) << 10;  // 2^(e-127) as fp16 (normal within the range above)
  return h | (h << 16);
}

__device__ __forceinline__ uint32_t e8m0_bf16x2(uint32_t e) {
  const uint32_t b = e ? (e << 7) : 0x0040u;  // 2^(e-127) in bf16 (e = 0 is the subnormal 2^-127)
  return b | (b << 16);
}

struct PfArgs {
  int H, I, k, S;
  int mode;           // 0: gate/up + SwiGLU, 1: down
  int K;              // reduction length (H or I)
  int tiles;          // feature tiles per item
  const int* xsig;    // mode 0: power-of-two exponent of each sorted row of the fp16 activation copy
  int allow_f16;      // mode 0: tiles whose scales all lie in the fp16 range run as fp16 MMAs
  const uint8_t* sc0; // E8M0 scales of the first matrix (w1 or w2) of slot 0; slot s at + s * B
  const uint8_t* sc1; // E8M0 scales of w3 (mode 0)
  size_t B;           // bytes per expert
  const PfItem* items;
  const int* n_items;
  const int* perm;    // sorted position -> pair index (mode 1 epilogue)
  __nv_bfloat16* hs;  // mode 0 output [P, I]
  float* o;           // mode 1 output [P, H] by pair
  int* err;
  // row-scaled FP8 weights (the shared expert): per-row fp32 scales of w1 and
  // w3 (mode 0) or w2 (mode 1); items are the row ranges [64 i, 64 i + 64) of
  // `rows` rows, and mode 1 writes row r of the output at o[(o_row0 + r) * H]
  const float* rs0;
  const float* rs1;
  int rows;
  int o_row0;
  int mx;             // mode 0: h quantised to MXFP4 along I (blocks of 32 features) before the store
  const int8_t* slot_part;  // non-null: only items whose slot_part[slot] == part_sel run
  int part_sel;
};

// FP8 = false: MXFP4 experts of the slot pool (E2M1 codes with E8M0 block
// scales), items from the grouped pair list.  FP8 = true: one row-scaled E4M3
// matrix pair (the shared expert) over all tokens: codes are read 64 bytes
// per row per K step, decoded exactly to fp16 (mode 0) or bf16 (mode 1), and
// the row scales are applied to the fp32 accumulators.
template <class C, bool FP8>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_gemm_kernel(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
                        const __grid_constant__ CUtensorMap mB, const __grid_constant__ CUtensorMap mB16,
                        PfArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bar = (uint64_t*)(sm + C::kOffBar);
  uint64_t* full = bar;                    // [C::kStages]
  uint64_t* empty = bar + C::kStages;      // [C::kStages]
  uint64_t* rawf = bar + 2 * C::kStages;   // [C::kRaw]
  uint64_t* rawe = rawf + C::kRaw;       // [C::kRaw]
  uint64_t* done = rawe + C::kRaw;
  uint32_t* tmem_slot = (uint32_t*)(done + 1);
  int* f16_flag = (int*)(tmem_slot + 1);
  // raw-code ring: FP8 rows take twice the bytes per K step, in half as many stages
  constexpr int kRT = FP8 ? 2 * kRawTile : kRawTile;
  constexpr int kRing = FP8 ? C::kRaw / 2 : C::kRaw;
  // TMA fills may land out of order.  A group's own earlier waits imply that
  // the previous fill of a raw slot (step ks - kRing) has landed when kRing is
  // a multiple of the group count (the group converted it itself) or when
  // kRing >= kStages + groups (its previous step waited for the MMA of step
  // ks - 3 - kStages, which needed step ks - kRing converted); otherwise it
  // first waits for that fill's conversion on rawe, so that rawf's parity
  // cannot pass on the older phase.
  constexpr bool kRawGuard = kRing % kPfConvGroups != 0 && kRing < C::kStages + kPfConvGroups;
  constexpr int kRowB = FP8 ? 64 : 32;  // code bytes per weight row per K step

  const int item_idx = blockIdx.x / a.tiles;
  const int tile = blockIdx.x % a.tiles;
  PfItem it;
  if (FP8) {
    it.slot = 0;
    it.row0 = item_idx * C::kNMax;
    it.count = min(C::kNMax, a.rows - it.row0);
    it.pad = 0;
    if (it.count < 1) return;
  } else {
    if (item_idx >= *a.n_items) return;
    it = a.items[item_idx];
    if (a.slot_part && (it.slot < 0 || it.slot >= a.S || a.slot_part[it.slot] != a.part_sel)) return;
  }
  if (it.count > C::kNMax || it.count < 1) {  // the host picks the shape from T; never expected
    if (threadIdx.x == 0) atomicCAS(a.err, 0, MOE_ERR_INVALID);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = a.K / kPfKStep;
  const int sbytes = a.K / 32;                   // scale bytes per weight row
  const int n_mma = (it.count + 15) & ~15;       // MMA N
  const int n_box = (it.count + kPfBox - 1) / kPfBox;
  const uint32_t b_bytes = (uint32_t)n_box * kPfBox * 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], kPfConvThreads + 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&rawf[s], 1);
      mbar_init(&rawe[s], kPfConvThreads);
    }
    mbar_init(done, 1);
    // E4M3 values are exact in fp16 (gate/up runs against the fp16 activation copy)
    *f16_flag = (a.mode == 0 && (FP8 || a.allow_f16)) ? 1 : 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kWarpMma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // first weight row of this CTA: mode 0 -> feature f0 of w1 (tile 0) and of
  // w3 (tile 1), 128 features each; mode 1 -> row f0 of w2 (256 rows)
  const int f0 = a.mode == 0 ? tile * 128 : tile * 256;

  // fp16 or bf16 operands for this tile: fp16 when every block scale of the
  // tile keeps the scaled E2M1 values exact in fp16 (gate/up only).  The vote
  // runs in every warp but the raw-code producer, which starts streaming at once.
  bool f16 = false;
  if (warp != kWarpRaw) {
    if (!FP8 && a.mode == 0 && a.allow_f16 && warp < 8) {
      const int r = threadIdx.x >> 1, c = threadIdx.x & 1;
      const int g = r & 1, i = r >> 1;
      uint4 q[kPfMT][4];
#pragma unroll
      for (int mt = 0; mt < kPfMT; ++mt) {
        const uint8_t* row = (g ? a.sc1 : a.sc0) + (size_t)it.slot * a.B + (size_t)(f0 + 64 * mt + i) * sbytes;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int off = c * 16 + j * 32;
          q[mt][j] = off < sbytes ? __ldg(reinterpret_cast<const uint4*>(row + off))
                                  : make_uint4(0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu);
        }
      }
      bool in_range = true;
#pragma unroll
      for (int mt = 0; mt < kPfMT; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t w4[4] = {q[mt][j].x, q[mt][j].y, q[mt][j].z, q[mt][j].w};
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              const uint32_t e = (w4[u] >> (8 * b)) & 0xff;
              in_range = in_range && e >= kF16ScaleLo && e <= kF16ScaleHi;
            }
        }
      if (!in_range) atomicAnd(f16_flag, 0);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kPfThreads - 32) : "memory");
    f16 = *(volatile int*)f16_flag != 0;
  }

  if (warp == kWarpRaw) {
    // weight codes: as far ahead as the raw ring allows, independent of MMA progress
    if (lane == 0) {
      bool ok = true;
      for (int rk = 0; rk < nk && ok; ++rk) {
        const int rs = rk % kRing, rr = rk / kRing;
        if (rr > 0) ok = mbar_wait_fast(&rawe[rs], (rr - 1) & 1, a.err);
        if (!ok) break;
        uint8_t* dst = sm + C::kOffRaw + rs * kRT;
        mbar_expect_tx(&rawf[rs], kRT);
        if (FP8) {  // 2-D maps over one matrix: (row bytes, rows)
          if (a.mode == 0) {
            tma_2d(dst, &mA0, rk * 64, f0, &rawf[rs]);
            tma_2d(dst + 128 * 64, &mA1, rk * 64, f0, &rawf[rs]);
          } else {
            tma_2d(dst, &mA0, rk * 64, f0, &rawf[rs]);
          }
        } else if (a.mode == 0) {
          tma_3d(dst, &mA0, rk * 32, f0, it.slot, &rawf[rs]);
          tma_3d(dst + 128 * 32, &mA1, rk * 32, f0, it.slot, &rawf[rs]);
        } else {
          tma_3d(dst, &mA0, rk * 32, f0, it.slot, &rawf[rs]);
        }
      }
      if (!ok) {  // let copies already issued land before the CTA can exit
        const uint64_t t0 = gtimer();
        while (gtimer() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == kWarpB) {
    // activation tiles: one stage per free operand slot
    if (lane == 0) {
      bool ok = true;
      for (int ks = 0; ks < nk && ok; ++ks) {
        const int s = ks % C::kStages, r = ks / C::kStages;
        if (r > 0) ok = mbar_wait_fast(&empty[s], (r - 1) & 1, a.err);
        if (!ok) break;
        uint8_t* bdst = sm + C::kOffB + s * C::kBTile;
        mbar_expect_tx(&full[s], b_bytes);
        for (int bx = 0; bx < n_box; ++bx)
          tma_2d(bdst + bx * kPfBox * 128, f16 ? &mB16 : &mB, ks * kPfKStep, it.row0 + bx * kPfBox, &full[s]);
      }
      if (!ok) {
        const uint64_t t0 = gtimer();
        while (gtimer() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == kWarpMma) {
    // the whole warp runs the loop and one elected lane issues: operands stay
    // warp-uniform, and a K step's MMAs and commit go out as one block
    const uint32_t idesc = idesc_16bit(n_mma, !f16);
    bool ok = true;
    for (int ks = 0; ks < nk && ok; ++ks) {
      const int s = ks % C::kStages, r = ks / C::kStages;
      ok = __all_sync(0xffffffffu, mbar_wait_fast(&full[s], r & 1, a.err));
      if (!ok) break;
      tc_fence_after();
      const uint64_t bd = umma_desc_sw128(su32(sm + C::kOffB + s * C::kBTile));
      const uint64_t a0 = umma_desc_sw128(su32(sm + C::kOffA + s * kAStage));
      const uint64_t a1 = umma_desc_sw128(su32(sm + C::kOffA + s * kAStage + kATile));
      static_assert(kPfMT == 2 && kPfKStep == 64, "mma_kstep_2x4 covers two tiles x four K = 16 slices");
      mma_kstep_2x4(tmem, tmem + 256u, a0, a1, bd, idesc, ks != 0, &empty[s]);
    }
    mma_commit_elect(done);  // fires when every issued MMA has completed
  } else if (warp < kPfConvWarps) {
    // converters: group cg takes the K steps ks = cg (mod 3); thread -> row r
    // of both 128 x 64 A tiles (two 32-weight halves each)
    const int cg = warp / (kPfConvThreads / 32);
    const int r = threadIdx.x & (kPfConvThreads - 1);
    int raw_off[kPfMT];
    const uint8_t* srow[kPfMT];
#pragma unroll
    for (int mt = 0; mt < kPfMT; ++mt) {
      if (a.mode == 0) {  // tile 0: w1 row f0 + r (gate), tile 1: w3 row f0 + r (up)
        raw_off[mt] = mt * (128 * kRowB) + r * kRowB;
        srow[mt] = FP8 ? nullptr : (mt ? a.sc1 : a.sc0) + (size_t)it.slot * a.B + (size_t)(f0 + r) * sbytes;
      } else {
        raw_off[mt] = (128 * mt + r) * kRowB;
        srow[mt] = FP8 ? nullptr : a.sc0 + (size_t)it.slot * a.B + (size_t)(f0 + 128 * mt + r) * sbytes;
      }
    }
    // scale bytes: 16 at a time (8 K steps), loaded one group ahead
    uint4 scur[kPfMT], snext[kPfMT];
#pragma unroll
    for (int mt = 0; mt < kPfMT; ++mt) {
      if (FP8) {
        scur[mt] = snext[mt] = make_uint4(0, 0, 0, 0);
      } else {
        scur[mt] = __ldg(reinterpret_cast<const uint4*>(srow[mt]));
        snext[mt] = sbytes > 16 ? __ldg(reinterpret_cast<const uint4*>(srow[mt] + 16)) : scur[mt];
      }
    }
    bool ok = true;
    int chunk = 0;  // scur holds the scale bytes of K steps 8 * chunk .. 8 * chunk + 7
    for (int ks = cg; ks < nk && ok; ks += kPfConvGroups) {
      const int rs = ks % kRing, rr = ks / kRing;
      const int s = ks % C::kStages, rnd = ks / C::kStages;
      if (!FP8 && ks / 8 != chunk) {  // a stride below 8 moves on by one chunk at a time
        ++chunk;
#pragma unroll
        for (int mt = 0; mt < kPfMT; ++mt) {
          scur[mt] = snext[mt];
          const int nxt = (chunk + 1) * 16;
          if (nxt < sbytes) snext[mt] = __ldg(reinterpret_cast<const uint4*>(srow[mt] + nxt));
        }
      }
      if (kRawGuard && rr > 0 && !(ok = mbar_wait_fast(&rawe[rs], (rr - 1) & 1, a.err))) break;
      if (!(ok = mbar_wait_fast(&rawf[rs], rr & 1, a.err))) break;
      if (FP8) {
        // 64 E4M3 codes per row: exact 16-bit values, no block scale
        uint4 q8[kPfMT][4];
#pragma unroll
        for (int mt = 0; mt < kPfMT; ++mt)
#pragma unroll
          for (int c = 0; c < 4; ++c)
            q8[mt][c] = *reinterpret_cast<const uint4*>(sm + C::kOffRaw + rs * kRT + raw_off[mt] + 16 * c);
        if (rnd > 0 && !(ok = mbar_wait_fast(&empty[s], (rnd - 1) & 1, a.err))) {
          mbar_arrive(&rawe[rs]);
          break;
        }
#pragma unroll
        for (int mt = 0; mt < kPfMT; ++mt) {
          uint8_t* arow = sm + C::kOffA + s * kAStage + mt * kATile + r * 128;
#pragma unroll
          for (int unit = 0; unit < 8; ++unit) {  // 8 weights = two code words
            const uint4 v = q8[mt][unit >> 1];
            const uint32_t w0 = (unit & 1) ? v.z : v.x, w1 = (unit & 1) ? v.w : v.y;
            uint4 o;
            fp8x4_to_f16(w0, o.x, o.y);
            fp8x4_to_f16(w1, o.z, o.w);
            if (!f16) {
              o.x = f16x2_to_bf16x2(o.x);
              o.y = f16x2_to_bf16x2(o.y);
              o.z = f16x2_to_bf16x2(o.z);
              o.w = f16x2_to_bf16x2(o.w);
            }
            *reinterpret_cast<uint4*>(arow + ((unit ^ (r & 7)) << 4)) = o;
          }
        }
      } else {
        uint4 q[kPfMT][2];
#pragma unroll
        for (int mt = 0; mt < kPfMT; ++mt) {
          const uint8_t* src = sm + C::kOffRaw + rs * kRT + raw_off[mt];
          q[mt][0] = *reinterpret_cast<const uint4*>(src);
          q[mt][1] = *reinterpret_cast<const uint4*>(src + 16);
        }
        if (rnd > 0 && !(ok = mbar_wait_fast(&empty[s], (rnd - 1) & 1, a.err))) {
          mbar_arrive(&rawe[rs]);
          break;
        }
#pragma unroll
        for (int mt = 0; mt < kPfMT; ++mt) {
          uint8_t* arow = sm + C::kOffA + s * kAStage + mt * kATile + r * 128;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int sb = (ks & 7) * 2 + c;  // scale byte within the 16 loaded
            const uint32_t sw = sb < 4 ? scur[mt].x : sb < 8 ? scur[mt].y : sb < 12 ? scur[mt].z : scur[mt].w;
            const uint32_t e8 = (sw >> (8 * (sb & 3))) & 0xff;
            const uint32_t sc2 = f16 ? e8m0_f16x2(e8) : e8m0_bf16x2(e8);
            const uint32_t w4[4] = {q[mt][c].x, q[mt][c].y, q[mt][c].z, q[mt][c].w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              uint4 o;
              fp4x8_to_f16(w4[u], o.x, o.y, o.z, o.w);
              if (f16) {
                o.x = hmul2_f16(o.x, sc2);
                o.y = hmul2_f16(o.y, sc2);
                o.z = hmul2_f16(o.z, sc2);
                o.w = hmul2_f16(o.w, sc2);
              } else {
                o.x = f16x2_to_bf16x2_scaled(o.x, sc2);
                o.y = f16x2_to_bf16x2_scaled(o.y, sc2);
                o.z = f16x2_to_bf16x2_scaled(o.z, sc2);
                o.w = f16x2_to_bf16x2_scaled(o.w, sc2);
              }
              const int unit = c * 4 + u;
              *reinterpret_cast<uint4*>(arow + ((unit ^ (r & 7)) << 4)) = o;
            }
          }
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(&full[s]);
      // the raw stage is released only now: its codes have been used, so the
      // shared-memory loads are complete before the next TMA can overwrite it
      // (an arrive right after issuing the loads let the refill overtake them)
      mbar_arrive(&rawe[rs]);
    }
  }

  // epilogue: all 16 warps.  Warp w reads TMEM lane quadrant w % 4 and takes
  // every fourth 16-column chunk (w / 4 picks which): gate/up reads the same
  // chunk of both accumulators (gate and up of feature f0 + row), down each
  // accumulator's chunks in turn.
  {
    __syncwarp();
    // the raw-code producer warp did not take part in the vote: it reads the
    // result once the MMAs are done; the other warps load the per-column
    // values of their chunks (the activation copy's row exponents, or the
    // pair of each column) before they wait
    bool ok = true;
    if (warp == kWarpRaw) {
      ok = __all_sync(0xffffffffu, mbar_wait(done, 0, a.err));
      __syncwarp();
      f16 = *(volatile int*)f16_flag != 0;
    }
    const int q = warp & 3, part = warp >> 2;
    const int row = q * 32 + lane;  // D row = A tile row
    const int nchunks = n_mma / 16;
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
    constexpr int kParts = kPfWarps / 4;
    if (a.mode == 0) {
      constexpr int kMaxChunks = (C::kNMax / 16 + kParts - 1) / kParts;
      static_assert(kMaxChunks <= 4, "one word of packed exponents");
      const int feat = f0 + row;
      const float rg = FP8 ? a.rs0[feat] : 1.f, ru = FP8 ? a.rs1[feat] : 1.f;
      // chunk i's exponent (|e| < 128) for column c0 + j in byte i of lane j
      uint32_t sgw = 0;
#pragma unroll
      for (int i = 0; i < kMaxChunks; ++i) {
        const int cl = part * 16 + i * kParts * 16 + (lane & 15);
        const uint32_t e = (f16 && cl < it.count) ? ((uint32_t)a.xsig[it.row0 + cl] & 0xffu) : 0u;
        sgw |= e << (8 * i);
      }
      if (warp != kWarpRaw) {
        ok = __all_sync(0xffffffffu, mbar_wait(done, 0, a.err));
        __syncwarp();
      }
      tc_fence_after();
#pragma unroll 1
      for (int i = 0; ok && i < kMaxChunks; ++i) {
        const int c0 = part * 16 + i * kParts * 16;
        if (c0 >= n_mma) break;
        const int sg = (int)(sgw << (24 - 8 * i)) >> 24;
        uint32_t vg[16], vu[16];
        tmem_ld16_nw(tq + (uint32_t)c0, vg);
        tmem_ld16_nw(tq + (uint32_t)(256 + c0), vu);
        tmem_ld_wait16(vg);
        tmem_ld_fence16(vu);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int col = c0 + j;
          const float sc = __uint_as_float((uint32_t)(127 + __shfl_sync(0xffffffffu, sg, j)) << 23);
          if (col < it.count) {
            // SiLU(g) = g * sigmoid(g) with sigmoid(g) = (1 + tanh(g / 2)) / 2: one
            // hardware tanh (relative error ~2^-11, below h's bf16 rounding)
            const float hg = 0.5f * __uint_as_float(vg[j]) * (sc * rg), up = __uint_as_float(vu[j]) * (sc * ru);
            float hv = fmaf(hg, tanh_approx(hg), hg) * up;
            if (a.mx) {
              // the warp's 32 lanes hold 32 consecutive features of this column: one MX block
              const uint32_t amax = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(hv)));
              const uint32_t sb = mx_scale_byte(__uint_as_float(amax));
              hv = mx_value(mx_code(hv, mx_inv_scale(sb)), mx_scale(sb));
            }
            a.hs[(size_t)(it.row0 + col) * a.I + feat] = __float2bfloat16_rn(hv);
          }
        }
      }
    } else {
      constexpr int kMaxChunks = (kPfMT * C::kNMax / 16 + kParts - 1) / kParts;
      static_assert(kPfMT == 2, "two row scales");
      const float rw0 = FP8 ? a.rs0[f0 + row] : 1.f, rw1 = FP8 ? a.rs0[f0 + 128 + row] : 1.f;
      int plv[kMaxChunks];  // lane j < 16: the output row of column c0 + j of chunk i
#pragma unroll
      for (int i = 0; i < kMaxChunks; ++i) {
        const int cc = part + i * kParts;
        const int cl = (nchunks > 0 ? cc % nchunks : 0) * 16 + (lane & 15);
        plv[i] = (cc < kPfMT * nchunks && cl < it.count) ? (FP8 ? a.o_row0 + it.row0 + cl : a.perm[it.row0 + cl]) : 0;
      }
      if (warp != kWarpRaw) {
        ok = __all_sync(0xffffffffu, mbar_wait(done, 0, a.err));
        __syncwarp();
      }
      tc_fence_after();
#pragma unroll
      for (int i = 0; i < kMaxChunks; ++i) {
        const int cc = part + i * kParts;
        if (!ok || cc >= kPfMT * nchunks) break;
        const int mt = cc / nchunks, c0 = (cc % nchunks) * 16;
        uint32_t v[16];
        tmem_ld16(tq + (uint32_t)(mt * 256 + c0), v);
        const int feat = f0 + 128 * mt + row;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int p = __shfl_sync(0xffffffffu, plv[i], j);
          if (c0 + j < it.count) a.o[(size_t)p * a.H + feat] = __uint_as_float(v[j]) * (mt ? rw1 : rw0);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
  }
}

// ------------------------------------------- block-scaled FP4 (kind::mxf4) --
// The A-quantised mode (activations quantised to MXFP4 by the OCP MX rule, as
// the weights are): both operands are E2M1 codes with one E8M0 scale per 32
// elements, multiplied by tcgen05.mma.kind::mxf4.block_scale.  The packed codes
// go from global memory to shared memory by TMA (128-byte swizzle, 256 codes per
// row and stage) with no conversion; the scale factors go to tensor memory.
//
// Tensor-memory layout of the scale factors (measured with a one-MMA probe on
// sm_103a): the tensor core computes D rows 32 q .. 32 q + 31 in lane quadrant
// q and takes their scales from that quadrant's lanes.  Per 128-K window (four
// 32-element blocks, two K = 64 MMAs with scale-factor IDs 0 and 2) a 4-column
// group holds, for A, row m's four block scales (bytes 0..3) in lane m, column
// group + m / 32; for B, row n's in lane 32 q + n % 32, column group + n / 32 of
// every quadrant q.
constexpr int kMxThreads = 512;   // warp 0 TMA, warp 1 MMA, warps 4-7 scale factors, warps 4-15 the epilogue
constexpr int kMxEpiWarps = kMxThreads / 32 - 4;  // three per tensor-memory lane quadrant
constexpr int kMxEpiParts = kMxEpiWarps / 4;
constexpr int kMxQueue = 4;       // work indices published ahead to the consumer warps
constexpr int kMxStages = 3;      // shared-memory stages of codes
constexpr int kMxSfSlots = 2;     // tensor-memory slots of scale factors (stage ks in slot ks % 2)
constexpr int kMxKStage = 256;    // K elements per stage: one 128-byte row of packed codes
constexpr int kMxATile = 128 * 128;
constexpr int kMxAStage = 2 * kMxATile;
constexpr int kMxBStage = 256 * 128;  // up to four 64-row boxes
constexpr int kMxOffB = kMxStages * kMxAStage;
constexpr int kMxOffBar = kMxOffB + kMxStages * kMxBStage;
constexpr int kMxOffH = kMxOffBar + 256;          // gate/up: an item's h codes and scales before they go out
constexpr int kMxHRow = 80;                        // per row: 128 features' codes, their 4 scale bytes, pad to 16 B
static_assert(kMxHRow % 16 == 0 && kMxHRow >= 64 + 4, "staged h rows are read 16 bytes at a time");
constexpr int kMxSmem = kMxOffH + kMxNMax * kMxHRow + 1024;
static_assert(kMxSmem <= 232448, "shared memory per CTA");
constexpr int kMxSfBase = 2 * kMxNMax;  // first scale-factor column (after the two accumulators)
// per scale slot, 32 columns at kMxSfBase + 32 slot: A tile 0 (windows 0, 1) +0,
// +4; A tile 1 +8, +12; B window 0 +16 .. +22, window 1 +24 .. +30
static_assert(kMxSfBase + 32 * kMxSfSlots <= 512, "tensor memory columns");
static_assert(kMxNMax % 32 == 0 && kMxNMax / 32 <= 8 && kMxNMax <= 256, "B scale columns per window");
static_assert((2 * kMxStages + 4 + 2 * kMxQueue) * 8 + 8 + 4 * kMxQueue <= 256, "barrier area");

struct MxArgs {
  int mode;            // 0: gate/up + SwiGLU, h quantised to MXFP4; 1: down
  int K;               // reduction length (H or I)
  int tiles;           // feature tiles per item
  int H, I, S, P;
  size_t B;            // bytes per expert
  const uint8_t* sc0;  // E8M0 scales of w1 (mode 0) or w2 (mode 1) of slot 0 (slot s at + s * B)
  const uint8_t* sc1;  // w3 scales (mode 0)
  const uint8_t* bsc;  // E8M0 scales of the activation rows [P][K / 32] (sorted order)
  const PfItem* items;
  const int* n_items;
  int max_items;       // capacity of the item list
  int* ctr;            // work counter (zeroed by the item kernel): work past the first gridDim.x is drawn from it
  const int* perm;     // sorted position -> pair index (mode 1 output rows)
  uint8_t* hq;         // mode 0 out: h codes [P][I / 2]
  uint8_t* hsc;        // mode 0 out: h scales [P][I / 32]
  float* o;            // mode 1 out: [P][H] by pair
  int* err;
};

// One stage (K = 256) of both tiles: four K = 64 MMAs per tile, scale windows
// 0 (IDs 0, 2) then 1 (IDs 0, 2); descriptors advance 32 bytes (+2) per MMA.
__device__ __forceinline__ void mma_mx_stage(uint32_t d0, uint32_t d1, uint64_t a0, uint64_t a1, uint64_t b,
                                             uint32_t id0, uint32_t id2, uint32_t sf, uint32_t acc, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t.reg .b64 a, bb;\n\t.reg .b32 sa0, sa1, sb;\n\t"
      "elect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %8, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
      // window 0
      "add.u32 sa0, %7, 0;\n\tadd.u32 sa1, %7, 8;\n\tadd.u32 sb, %7, 16;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.block32 [%0], %2, %4, %5, [sa0], [sb], p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.block32 [%1], %3, %4, %5, [sa1], [sb], p;\n\t"
      "add.s64 a, %2, 2;\n\tadd.s64 bb, %4, 2;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.block32 [%0], a, bb, %6, [sa0], [sb], t;\n\t"
      "add.s64 a, %3, 2;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.block32 [%1], a, bb, %6, [sa1], [sb], t;\n\t"
      // window 1
      "add.u32 sa0, %7, 4;\n\tadd.u32 sa1, %7, 12;\n\tadd.u32 sb, %7, 24;\n\t"
      "add.s64 a, %2, 4;\n\tadd.s64 bb, %4, 4;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.block32 [%0], a, bb, %5, [sa0], [sb], t;\n\t"
      "add.s64 a, %3, 4;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.block32 [%1], a, bb, %5, [sa1], [sb], t;\n\t"
      "add.s64 a, %2, 6;\n\tadd.s64 bb, %4, 6;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.block32 [%0], a, bb, %6, [sa0], [sb], t;\n\t"
      "add.s64 a, %3, 6;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.block32 [%1], a, bb, %6, [sa1], [sb], t;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%9];\n\t}" ::"r"(d0),
      "r"(d1), "l"(a0), "l"(a1), "l"(b), "r"(id0), "r"(id2), "r"(sf), "r"(acc), "r"(su32(bar))
      : "memory");
}

// Block-scaled FP4 grouped GEMM, persistent (one CTA per SM): each work unit
// (item, feature tile) of mode 0 computes 128 features' gate (w1) and up (w3)
// rows over K = H and writes h = SiLU(gate) * up quantised to MXFP4 along I;
// of mode 1, 256 rows of w2 over K = I, written as fp32 outputs per pair.  CTA c
// starts with unit c and draws the next from a counter the item kernel zeroes;
// warp 0 publishes each to the other warps through a queue in shared memory and
// loads the next unit's stages while the current one's epilogue runs.
__global__ void __launch_bounds__(kMxThreads, 1)
    mxf4_gemm_kernel(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
                     const __grid_constant__ CUtensorMap mB, MxArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full = (uint64_t*)(sm + kMxOffBar);  // [kMxStages]: TMA bytes + four scale-factor warps
  uint64_t* empty = full + kMxStages;             // [kMxStages]: the stage's MMAs completed
  uint64_t* accf = empty + kMxStages;             // the item's MMAs completed
  uint64_t* acce = accf + 1;                      // the epilogue warps have read the accumulators
  uint64_t* drain = acce + 1;
  uint64_t* qfull = drain + 1;                    // [kMxQueue]: an item index published
  uint64_t* qempty = qfull + kMxQueue;            // [kMxQueue]: the MMA warp and the epilogue warps have read it
  uint64_t* esync = qempty + kMxQueue;            // the epilogue warps meet (h staging)
  uint32_t* tmem_slot = (uint32_t*)(esync + 1);
  volatile int* itq = (volatile int*)(tmem_slot + 1);  // [kMxQueue] work indices, -1 = no more
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = a.K / kMxKStage;
  const int sbytes = a.K / 32;  // scale bytes per row
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (const CUtensorMap* m : {&mA0, &mA1, &mB})
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
    for (int s = 0; s < kMxStages; ++s) {
      mbar_init(&full[s], 1 + 4);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accf, 1);
    mbar_init(acce, kMxEpiWarps);
    mbar_init(drain, 1);
    for (int j = 0; j < kMxQueue; ++j) {
      mbar_init(&qfull[j], 1);
      mbar_init(&qempty[j], 1 + kMxEpiWarps);
    }
    mbar_init(esync, kMxEpiWarps);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // launched early: the items, activations and counters come from the kernels before
  int n_it = *a.n_items;
  if (n_it < 0 || n_it > a.max_items) {
    if (threadIdx.x == 0) atomicCAS(a.err, 0, MOE_ERR_INVALID);
    n_it = 0;
  }
  const int n_work = n_it * a.tiles;
  // work index -> (item, feature tile); an item the item kernel never produces
  // is skipped by every role (and flagged by the MMA warp)
  struct Work {
    PfItem it;
    int f0, n_mma, n_box;
    bool run;
  };
  auto work = [&](int w, bool flag) -> Work {
    Work r;
    r.it = a.items[w / a.tiles];
    const int tile = w % a.tiles;
    r.run = !(r.it.count < 1 || r.it.count > kMxNMax || r.it.slot < 0 || r.it.slot >= a.S || r.it.row0 < 0 ||
              r.it.row0 + r.it.count > a.P);
    if (!r.run && flag) atomicCAS(a.err, 0, MOE_ERR_INVALID);
    r.f0 = a.mode == 0 ? tile * 128 : tile * 256;
    r.n_mma = (r.it.count + 15) & ~15;
    r.n_box = (r.it.count + 63) / 64;
    return r;
  };
  // q-th work index of this CTA for a consumer warp (whole warp): false on timeout
  auto next_work = [&](uint32_t q, int& w) -> bool {
    const int j = q % kMxQueue;
    if (!__all_sync(0xffffffffu, mbar_wait_fast(&qfull[j], (q / kMxQueue) & 1, a.err))) return false;
    w = itq[j];
    __syncwarp();
    if (lane == 0) mbar_arrive(&qempty[j]);
    return true;
  };

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      uint32_t gs = 0, q = 0;
      auto publish = [&](int w) -> bool {
        const int j = q % kMxQueue;
        const uint32_t r = q / kMxQueue;
        if (r > 0 && !mbar_wait_fast(&qempty[j], (r - 1) & 1, a.err)) return false;
        itq[j] = w;
        mbar_arrive(&qfull[j]);  // release: the index is visible to the warps that wait on it
        ++q;
        return true;
      };
      int cur = (int)blockIdx.x < n_work ? (int)blockIdx.x : -1;
      ok = publish(cur);
      while (ok && cur >= 0) {
        const int ticket = atomicAdd(a.ctr, 1);  // the next work index; its latency overlaps these loads
        const Work m = work(cur, false);
        if (m.run) {
          const uint32_t b_bytes = (uint32_t)m.n_box * 64 * 128;
          for (int ks = 0; ks < nk; ++ks, ++gs) {
            const int s = gs % kMxStages;
            const uint32_t r = gs / kMxStages;
            if (r > 0 && !(ok = mbar_wait_fast(&empty[s], (r - 1) & 1, a.err))) break;
            uint8_t* ad = sm + s * kMxAStage;
            uint8_t* bd = sm + kMxOffB + s * kMxBStage;
            mbar_expect_tx(&full[s], kMxAStage + b_bytes);
            const int x = ks * 128;  // byte column of the stage's codes (a multiple of 16)
            if (a.mode == 0) {
              tma_3d(ad, &mA0, x, m.f0, m.it.slot, &full[s]);
              tma_3d(ad + kMxATile, &mA1, x, m.f0, m.it.slot, &full[s]);
            } else {
              tma_3d(ad, &mA0, x, m.f0, m.it.slot, &full[s]);
              tma_3d(ad + kMxATile, &mA0, x, m.f0 + 128, m.it.slot, &full[s]);
            }
            for (int bx = 0; bx < m.n_box; ++bx) tma_2d(bd + bx * 64 * 128, &mB, x, m.it.row0 + bx * 64, &full[s]);
          }
        }
        if (!ok) break;
        int nxt = ticket + (int)gridDim.x;
        if (nxt >= n_work) nxt = -1;
        if (!(ok = publish(nxt))) break;
        cur = nxt;
      }
      if (!ok) {  // let copies already issued land before the CTA can exit
        const uint64_t t0 = gtimer();
        while (gtimer() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    bool ok = true;
    uint32_t gs = 0, i = 0;
    for (uint32_t qi = 0; ok; ++qi) {
      int w;
      if (!(ok = next_work(qi, w)) || w < 0) break;
      const Work m = work(w, true);
      if (!m.run) continue;
      // the epilogue of the previous item has read the accumulators
      if (i > 0 && !(ok = __all_sync(0xffffffffu, mbar_wait_fast(acce, (i - 1) & 1, a.err)))) break;
      ++i;
      tc_fence_after();
      // MXF4 x MXF4 -> fp32, M = 128, N = n_mma, both operands K-major; scale
      // factors E8M0; IDs 0 and 2 pick bytes 0-1 and 2-3 of a window's columns
      const uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(m.n_mma >> 3) << 17) | (1u << 23) |
                             ((uint32_t)(128 >> 4) << 24);
      const uint32_t id0 = idesc, id2 = idesc | (2u << 4) | (2u << 29);
      for (int ks = 0; ks < nk; ++ks, ++gs) {
        const int s = gs % kMxStages;
        const uint32_t r = gs / kMxStages;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait_fast(&full[s], r & 1, a.err)))) break;
        tc_fence_after();
        const uint64_t ad0 = umma_desc_sw128(su32(sm + s * kMxAStage));
        const uint64_t ad1 = umma_desc_sw128(su32(sm + s * kMxAStage + kMxATile));
        const uint64_t bd = umma_desc_sw128(su32(sm + kMxOffB + s * kMxBStage));
        mma_mx_stage(tmem, tmem + kMxNMax, ad0, ad1, bd, id0, id2, tmem + kMxSfBase + 32 * (gs % kMxSfSlots),
                     ks != 0, &empty[s]);
      }
      if (ok) mma_commit_elect(accf);
    }
    // every MMA this warp issued has completed before tensor memory is freed
    mma_commit_elect(drain);
    __syncwarp();
    mbar_wait(drain, 0, a.err);
  } else if (warp >= 4) {
    // warps 4-7: per item the scale factors of every stage into lane quadrant
    // q (warp 4 + q may write only lanes 32 q .. 32 q + 31), then part 0 of the
    // epilogue; warps 8-11 and 12-15: parts 1 and 2 of the epilogue (a part
    // takes every third chunk of columns)
    const int q = warp & 3, part = (warp - 4) >> 2;
    bool ok = true;
    uint32_t gs = 0, i = 0, nsync = 0;
    // the epilogue warps meet (bounded, so a warp that gave up cannot leave
    // the others waiting)
    auto epi_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(esync);
      return __all_sync(0xffffffffu, mbar_wait_fast(esync, (nsync++) & 1, a.err));
    };
    for (uint32_t qi = 0; ok; ++qi) {
      int w;
      if (!(ok = next_work(qi, w)) || w < 0) break;
      const Work m = work(w, false);
      if (!m.run) continue;
      const PfItem it = m.it;
      const int f0 = m.f0, n_mma = m.n_mma;
      if (part == 0) {
        const uint8_t* base_a = a.sc0 + (size_t)it.slot * a.B;
        const uint8_t* sa0 = base_a + (size_t)(f0 + 32 * q + lane) * sbytes;
        const uint8_t* sa1 = a.mode == 0 ? a.sc1 + (size_t)it.slot * a.B + (size_t)(f0 + 32 * q + lane) * sbytes
                                         : base_a + (size_t)(f0 + 128 + 32 * q + lane) * sbytes;
        const uint8_t* sb[kMxNMax / 32];
#pragma unroll
        for (int c = 0; c < kMxNMax / 32; ++c) {
          const int n = 32 * c + lane;
          sb[c] = a.bsc + (size_t)(it.row0 + (n < it.count ? n : 0)) * sbytes;  // rows past the item: any valid row
        }
        // a stage's scale words (per K window: A tile 0, A tile 1, B rows 32 c +
        // lane) are loaded two stages ahead of their tensor-memory writes,
        // through a ring of three register sets
        struct Sf {
          uint2 a0, a1, b[kMxNMax / 32];
        };
        auto load = [&](int ks, Sf& sf) {
          sf.a0 = __ldg(reinterpret_cast<const uint2*>(sa0 + 8 * ks));  // x: window 0, y: window 1
          sf.a1 = __ldg(reinterpret_cast<const uint2*>(sa1 + 8 * ks));
#pragma unroll
          for (int c = 0; c < kMxNMax / 32; ++c) sf.b[c] = __ldg(reinterpret_cast<const uint2*>(sb[c] + 8 * ks));
        };
        auto store = [&](const Sf& sf) -> bool {
          // the scale slot's previous stage (gs - kMxSfSlots) must have finished
          // its MMAs, whose commit arrived on that stage's "empty" barrier.  This
          // warp writes stage gs - 1's scales before stage gs's, and the MMAs of
          // a stage wait for its scales, so that barrier is at most one phase behind.
          const int p = (int)gs - kMxSfSlots;
          if (p >= 0 && !__all_sync(0xffffffffu, mbar_wait_fast(&empty[p % kMxStages], (p / kMxStages) & 1, a.err)))
            return false;
          uint32_t bw0[8], bw1[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            bw0[c] = c < kMxNMax / 32 ? sf.b[c < kMxNMax / 32 ? c : 0].x : 0u;
            bw1[c] = c < kMxNMax / 32 ? sf.b[c < kMxNMax / 32 ? c : 0].y : 0u;
          }
          const uint32_t col = tmem + ((uint32_t)(32 * q) << 16) + kMxSfBase + 32 * (gs % kMxSfSlots);
          tmem_st1(col + 0 + q, sf.a0.x);
          tmem_st1(col + 4 + q, sf.a0.y);
          tmem_st1(col + 8 + q, sf.a1.x);
          tmem_st1(col + 12 + q, sf.a1.y);
          tmem_st8(col + 16, bw0);
          tmem_st8(col + 24, bw1);
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[gs % kMxStages]);
          ++gs;
          return true;
        };
        Sf ring[3];
        load(0, ring[0]);
        if (nk > 1) load(1, ring[1]);
        for (int k0 = 0; k0 < nk && ok; k0 += 3) {
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            const int ks = k0 + j;
            if (ks >= nk || !ok) break;
            if (ks + 2 < nk) load(ks + 2, ring[(j + 2) % 3]);
            ok = store(ring[j]);
          }
        }
        if (!ok) break;
      }
      // epilogue: warp w reads TMEM lane quadrant w % 4; part p takes chunks
      // p, p + 3, ... of the columns (8 wide for gate/up, 16 for down)
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_fast(accf, i & 1, a.err)))) break;
      ++i;
      tc_fence_after();
      const int row = q * 32 + lane;
      const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
      if (a.mode == 0) {
        // lane = feature f0 + row: gate (w1 row) in tile 0, up (w3 row) in tile 1.
        // The 16 columns of a chunk go through each step together (independent
        // warp reductions and shuffles), so their latencies overlap.  The codes
        // and scales collect in shared memory (a row per token: 64 code bytes,
        // 4 scale bytes) and leave in 16-byte stores once every warp is done:
        // one narrow store per column and warp cost half the epilogue.
        uint8_t* hs = sm + kMxOffH;
        if (!(ok = epi_sync())) break;  // the previous item's rows have left
        for (int c0 = 8 * part; c0 < n_mma; c0 += 8 * kMxEpiParts) {
          uint32_t vg[8], vu[8];
          tmem_ld8_nw(tq + (uint32_t)c0, vg);  // both loads in flight, one wait
          tmem_ld8_nw(tq + (uint32_t)(kMxNMax + c0), vu);
          tmem_ld_wait8(vg);
          tmem_ld_fence8(vu);
          float hv[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float hg = 0.5f * __uint_as_float(vg[j]), up = __uint_as_float(vu[j]);
            hv[j] = fmaf(hg, tanh_approx(hg), hg) * up;
          }
          // the warp's 32 lanes hold 32 consecutive features of a column: one MX block
          uint32_t am[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) am[j] = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(hv[j])));
          uint32_t code[8], sbyte[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            sbyte[j] = mx_scale_byte(__uint_as_float(am[j]));
            code[j] = mx_code(hv[j], mx_inv_scale(sbyte[j]));
          }
          uint32_t hi[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) hi[j] = __shfl_down_sync(0xffffffffu, code[j], 1);
          // byte b of the block = codes of lanes 2b (low nibble) and 2b + 1
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint8_t* hr = hs + (c0 + j) * kMxHRow;
            if ((lane & 1) == 0) hr[16 * q + lane / 2] = (uint8_t)(code[j] | (hi[j] << 4));
            if (lane == 0) hr[64 + q] = (uint8_t)sbyte[j];
          }
        }
        // the accumulators are read: the next item's MMAs may start
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce);
        if (!(ok = epi_sync())) break;
        const int et = threadIdx.x - 128;  // over the epilogue warps
        for (int e = et; e < it.count * 4; e += 32 * kMxEpiWarps) {
          const int r = e >> 2, part = e & 3;
          *reinterpret_cast<uint4*>(a.hq + (size_t)(it.row0 + r) * (a.I / 2) + f0 / 2 + 16 * part) =
              *reinterpret_cast<const uint4*>(hs + r * kMxHRow + 16 * part);
        }
        for (int r = et; r < it.count; r += 32 * kMxEpiWarps)
          *reinterpret_cast<uint32_t*>(a.hsc + (size_t)(it.row0 + r) * (a.I / 32) + f0 / 32) =
              *reinterpret_cast<const uint32_t*>(hs + r * kMxHRow + 64);
        continue;
      } else {
        for (int mt = 0; mt < 2; ++mt) {
          const int feat = f0 + 128 * mt + row;
          for (int c0 = 16 * part; c0 < n_mma; c0 += 16 * kMxEpiParts) {
            uint32_t v[16];
            tmem_ld16(tq + (uint32_t)(mt * kMxNMax + c0), v);
            const int cl = c0 + (lane & 15);
            const int pl = cl < it.count ? a.perm[it.row0 + cl] : 0;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int p = __shfl_sync(0xffffffffu, pl, j);
              if (c0 + j < it.count) a.o[(size_t)p * a.H + feat] = __uint_as_float(v[j]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
  }
}

// One warp per sorted row: x of the pair's token quantised to MXFP4 (OCP MX,
// 32-element blocks along H): packed codes (element 2j in the low nibble of
// byte j) and one E8M0 scale byte per block.  Four lanes hold a block; H is a
// multiple of 256, so every lane takes part in every step.
__global__ void gather_mxq_kernel(const uint16_t* x, int H, int k, const int* perm, const int* offsets, int S,
                                  uint8_t* xq, uint8_t* xsc) {
  pdl_launch_dependents();  // the block-scaled GEMM sets itself up meanwhile
  const int n = offsets[S];
  const int lane = threadIdx.x & 31;
  const int units = H / 8;
  for (int i = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5); i < n;
       i += (int)((gridDim.x * (size_t)blockDim.x) >> 5)) {
    const int tok = perm[i] / k;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)tok * H);
    for (int c = lane; c < units; c += 32) {
      const uint4 v = src[c];
      float f[8];
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        f[2 * qq] = __uint_as_float(w4[qq] << 16);
        f[2 * qq + 1] = __uint_as_float(w4[qq] & 0xffff0000u);
      }
      float am = 0.f;
#pragma unroll
      for (int qq = 0; qq < 8; ++qq) am = fmaxf(am, fabsf(f[qq]));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
      const uint32_t sbyte = mx_scale_byte(am);
      const float inv = mx_inv_scale(sbyte);
      uint32_t word = 0;
#pragma unroll
      for (int qq = 0; qq < 8; ++qq) word |= mx_code(f[qq], inv) << (4 * qq);
      reinterpret_cast<uint32_t*>(xq + (size_t)i * (H / 2))[c] = word;
      if ((lane & 3) == 0) xsc[(size_t)i * (H / 32) + c / 4] = (uint8_t)sbyte;
    }
  }
}

// items: per slot, tiles of <= nmax sorted rows
__global__ void prefill_items_kernel(const int* offsets, int S, int nmax, PfItem* items, int* n_items) {
  __shared__ int ws[34];
  const int tid = threadIdx.x, NT = blockDim.x;
  const int per = (S + NT - 1) / NT;
  const int s0 = min(S, tid * per), s1 = min(S, s0 + per);
  int local = 0;
  for (int s = s0; s < s1; ++s) local += (offsets[s + 1] - offsets[s] + nmax - 1) / nmax;
  int total;
  int pos = block_exclusive_scan(local, ws, &total);
  for (int s = s0; s < s1; ++s) {
    const int b = offsets[s], cnt = offsets[s + 1] - b;
    for (int t = 0; t * nmax < cnt; ++t) {
      PfItem itm;
      itm.slot = s;
      itm.row0 = b + t * nmax;
      itm.count = min(nmax, cnt - t * nmax);
      itm.pad = 0;
      items[pos++] = itm;
    }
  }
  if (tid == 0) {
    n_items[0] = total;
    n_items[1] = 0;  // work counters of the persistent block-scaled GEMMs (gate/up, down)
    n_items[2] = 0;
  }
}

// One warp per sorted row: copy the token's bf16 row, and an fp16 copy scaled
// by the power of two that brings its largest magnitude into [1, 2).
// mx != 0: each 32-element block of the row is replaced by its MXFP4
// quantisation (exact in bf16); the fp16 copy is not written (bf16 MMAs only).
__global__ void gather_rows_kernel(const uint16_t* x, int H, int k, const int* perm, const int* offsets, int S,
                                   uint16_t* xg, __half* xg16, int* xsig, int mx) {
  const int n = offsets[S];
  const int lane = threadIdx.x & 31;
  const int units = H / 8;
  for (int i = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5); i < n;
       i += (int)((gridDim.x * (size_t)blockDim.x) >> 5)) {
    const int tok = perm[i] / k;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)tok * H);
    uint4* dst = reinterpret_cast<uint4*>(xg + (size_t)i * H);
    if (mx) {
      // units 4b .. 4b + 3 (one 32-element block) sit in four consecutive lanes;
      // H is a multiple of 256, so every lane takes part in every step
      for (int c = lane; c < units; c += 32) {
        const uint4 v = src[c];
        float f[8];
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          f[2 * q] = __uint_as_float(w4[q] << 16);
          f[2 * q + 1] = __uint_as_float(w4[q] & 0xffff0000u);
        }
        float am = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) am = fmaxf(am, fabsf(f[q]));
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
        const uint32_t sb = mx_scale_byte(am);
        const float inv = mx_inv_scale(sb), xs = mx_scale(sb);
        uint32_t o4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(mx_value(mx_code(f[2 * q], inv), xs)));
          const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(mx_value(mx_code(f[2 * q + 1], inv), xs)));
          o4[q] = lo | (hi << 16);
        }
        dst[c] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
      if (lane == 0) xsig[i] = 0;
      continue;
    }
    float m = 0.f;
    for (int c = lane; c < units; c += 32) {
      const uint4 v = src[c];
      dst[c] = v;
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w4[q] << 16)), fabsf(__uint_as_float(w4[q] & 0xffff0000u))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    int sg = 0;
    if (m > 0.f) {
      int e;
      frexpf(m, &e);
      sg = min(100, max(-100, e - 1));  // keeps 2^sg a normal float for the epilogue
    }
    if (lane == 0) xsig[i] = sg;
    __half* d16 = xg16 + (size_t)i * H;
    for (int c = lane; c < units; c += 32) {
      const uint4 v = src[c];
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
      __half2 hv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        hv[q] = __floats2half2_rn(ldexpf(__uint_as_float(w4[q] << 16), -sg),
                                  ldexpf(__uint_as_float(w4[q] & 0xffff0000u), -sg));
      reinterpret_cast<uint4*>(d16)[c] = *reinterpret_cast<uint4*>(hv);
    }
  }
}

// Four consecutive outputs per thread (16-byte loads of o, all k issued before
// use); per element the same fmaf chain in rank order.
__global__ void __launch_bounds__(256) prefill_combine_kernel(const float* o, const int32_t* slots, const float* w,
                                                              int T, int k, int H, int S, uint16_t* y) {
  const int t = blockIdx.y;
  for (int n = 4 * (blockIdx.x * blockDim.x + threadIdx.x); n < H; n += 4 * gridDim.x * blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int j = 0; j < k; ++j) {
      const int p = t * k + j;
      const int sl = slots[p];
      if (sl < 0 || sl >= S) continue;
      const float4 v = *reinterpret_cast<const float4*>(o + (size_t)p * H + n);
      const float wj = w[p];
      acc.x = fmaf(wj, v.x, acc.x);
      acc.y = fmaf(wj, v.y, acc.y);
      acc.z = fmaf(wj, v.z, acc.z);
      acc.w = fmaf(wj, v.w, acc.w);
    }
    uint2 out;
    out.x = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.x)) |
            ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.y)) << 16);
    out.y = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.z)) |
            ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.w)) << 16);
    uint16_t* dst = y + (size_t)t * H + n;
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

// ------------------------------------------------------------------- host --

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  });
  return fn;
}

// rank-3 byte map: (x: row bytes, y: rows, z: slots)
static moe_status map_bytes3(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint64_t slots,
                             uint64_t slot_stride, uint32_t box_x, uint32_t box_y) {
  auto fn = tensor_map_encoder();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {row_bytes, rows, slots};
  cuuint64_t strides[2] = {row_bytes, slot_stride};
  cuuint32_t box[3] = {box_x, box_y, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (weights) failed: %d", (int)r);
  return MOE_OK;
}

// rank-2 16-bit map (bf16 or fp16) with 128-byte swizzle, box 64 x kPfBox
static moe_status map_bf16_rows(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                                CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  auto fn = tensor_map_encoder();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kPfBox};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (activations) failed: %d", (int)r);
  return MOE_OK;
}

// Byte maps with 128-byte swizzle for packed FP4 codes: box of 128 bytes (256
// codes) by box_y rows.  Rank 3: (row bytes, rows, slots); rank 2: (row bytes, rows).
static moe_status map_codes_sw128(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows,
                                  uint64_t slots, uint64_t slot_stride, uint32_t box_y) {
  auto fn = tensor_map_encoder();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint32_t rank = slots ? 3 : 2;
  cuuint64_t dims[3] = {row_bytes, rows, slots ? slots : 1};
  cuuint64_t strides[2] = {row_bytes, slot_stride};
  cuuint32_t box[3] = {128, box_y, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (FP4 codes) failed: %d", (int)r);
  return MOE_OK;
}

moe_status group_pairs_multi(const int32_t* ids, int P, int E, int32_t* offsets, int32_t* perm, int32_t* d_error,
                             int* cnt_ws, cudaStream_t stream);
size_t group_pairs_multi_ws(int P, int E);

static size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

bool grouped_gemm_supported(const moe_expert_views* v) {
  return v && v->fp4_slots && v->fp4_num_slots >= 1 && v->fp4_num_slots <= 16384 && v->H % 512 == 0 &&
         v->I % 512 == 0;
}

size_t gg_index_bytes(int T, int k, int S) {
  const size_t P = (size_t)T * k;
  const size_t max_items = (size_t)S + P / kMxNMax + 1;  // the smaller items (block-scaled FP4 path)
  return a256((S + 1) * 4) + a256(P * 4) + a256(max_items * sizeof(PfItem)) + a256(16) +
         a256(group_pairs_multi_ws((int)P, S)) + a256(P * 4);
}

void gg_carve_index(uint8_t* base, int T, int k, int S, GgBufs* b) {
  const size_t P = (size_t)T * k;
  const size_t max_items = (size_t)S + P / kMxNMax + 1;
  size_t off = 0;
  b->offsets = (int*)(base + off);
  off += a256((S + 1) * 4);
  b->perm = (int*)(base + off);
  off += a256(P * 4);
  b->items = (PfItem*)(base + off);
  off += a256(max_items * sizeof(PfItem));
  b->nitems = (int*)(base + off);
  off += a256(16);
  b->cnt = (int*)(base + off);
  off += a256(group_pairs_multi_ws((int)P, S));
  b->xsig = (int*)(base + off);
}

moe_status grouped_gemm_fp4(const moe_expert_views* v, const uint16_t* x, int T, int k, const int32_t* slots,
                            const GgBufs& b, int32_t* d_error, cudaStream_t stream, const DownParts& down,
                            int mx_act) {
  const int H = v->H, I = v->I, S = v->fp4_num_slots;
  const size_t P = (size_t)T * k;
  moe_status st = group_pairs_multi(slots, (int)P, S, b.offsets, b.perm, d_error, b.cnt, stream);
  if (st != MOE_OK) return st;
  prefill_items_kernel<<<1, 1024, 0, stream>>>(b.offsets, S, kPfNMax, b.items, b.nitems);
  if ((st = check_launch("prefill_items_kernel")) != MOE_OK) return st;
  {
    const int blocks = (int)std::min<size_t>((P + 7) / 8, 152 * 16);
    gather_rows_kernel<<<blocks, 256, 0, stream>>>(x, H, k, b.perm, b.offsets, S, b.xg, b.xg16, b.xsig, mx_act);
    if ((st = check_launch("gather_rows_kernel")) != MOE_OK) return st;
  }
  // weight maps over the whole pool: dims (row bytes, rows, slots)
  const size_t B = fp4_bytes(H, I);
  const uint8_t* pool = v->fp4_slots;
  const size_t hi = (size_t)H * I;
  const uint8_t* w1c = pool;
  const uint8_t* w1s = pool + hi / 2;
  const uint8_t* w3c = pool + (hi / 2 + hi / 32);
  const uint8_t* w3s = w3c + hi / 2;
  const uint8_t* w2c = pool + 2 * (hi / 2 + hi / 32);
  const uint8_t* w2s = w2c + hi / 2;
  CUtensorMap m1c, m3c, m2c, mx, mx16, mh;
  if ((st = map_bytes3(&m1c, w1c, H / 2, I, S, B, 32, 128)) != MOE_OK) return st;
  if ((st = map_bytes3(&m3c, w3c, H / 2, I, S, B, 32, 128)) != MOE_OK) return st;
  if ((st = map_bytes3(&m2c, w2c, I / 2, H, S, B, 32, 256)) != MOE_OK) return st;
  if ((st = map_bf16_rows(&mx, b.xg, H, P)) != MOE_OK) return st;
  if ((st = map_bf16_rows(&mx16, b.xg16, H, P, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)) != MOE_OK) return st;
  if ((st = map_bf16_rows(&mh, b.hs, I, P)) != MOE_OK) return st;

  // items hold at most T rows (each token routes to a slot once): up to 64
  // tokens take the small shape (four operand stages)
  const bool small = T <= PfSmall::kNMax;
  {
    // a function attribute holds per device: set it on every call
    cudaError_t e = small ? cudaFuncSetAttribute(prefill_gemm_kernel<PfSmall, false>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, PfSmall::kSmem)
                          : cudaFuncSetAttribute(prefill_gemm_kernel<PfBig, false>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, PfBig::kSmem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prefill_gemm_kernel)");
  }
  // items: at most one per used slot, plus one per 256 further rows (wide shape)
  const int max_items = (int)std::min<size_t>((size_t)S, P) + (small ? 0 : (int)(P / kPfNMax) + 1);
  PfArgs pa{};
  pa.H = H;
  pa.I = I;
  pa.k = k;
  pa.S = S;
  pa.mx = mx_act;
  pa.items = b.items;
  pa.n_items = b.nitems;
  pa.perm = b.perm;
  pa.hs = b.hs;
  pa.o = b.o;
  pa.err = d_error;
  pa.B = B;
  pa.xsig = b.xsig;
  auto launch = [&](const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& bm, const CUtensorMap& bm16) {
    if (small)
      prefill_gemm_kernel<PfSmall, false><<<max_items * pa.tiles, kPfThreads, PfSmall::kSmem, stream>>>(a0, a1, bm, bm16, pa);
    else
      prefill_gemm_kernel<PfBig, false><<<max_items * pa.tiles, kPfThreads, PfBig::kSmem, stream>>>(a0, a1, bm, bm16, pa);
  };
  // GEMM1: gate/up, 128 features (their w1 rows and their w3 rows) per CTA
  pa.mode = 0;
  pa.K = H;
  pa.tiles = I / 128;
  pa.sc0 = w1s;
  pa.sc1 = w3s;
  pa.allow_f16 = mx_act ? 0 : 1;  // MXFP4 activations run as bf16 products (exact values)
  {
    ProfScope ps(MOE_K_GEMM_GATEUP, stream);
    launch(m1c, m3c, mx, mx16);
  }
  if ((st = check_launch("prefill_gemm_kernel (gate/up)")) != MOE_OK) return st;
  // GEMM2: down, 256 output features (two tiles of 128) per CTA; with parts,
  // one launch per part of the slots once that part's down matrices are in
  pa.mode = 1;
  pa.K = I;
  pa.tiles = H / 256;
  pa.sc0 = w2s;
  pa.sc1 = w2s;
  pa.allow_f16 = 0;
  const int np = down.n > 1 && down.slot_part ? down.n : 1;
  for (int q = 0; q < np; ++q) {
    const cudaEvent_t ev = down.n >= 1 && down.ready ? down.ready[np == 1 ? down.n - 1 : q] : nullptr;
    if (ev) MOE_CUDA(cudaStreamWaitEvent(stream, ev, 0));
    pa.slot_part = np > 1 ? down.slot_part : nullptr;
    pa.part_sel = q;
    {
      ProfScope ps(MOE_K_GEMM_DOWN, stream);
      launch(m2c, m2c, mh, mh);
    }
    if ((st = check_launch("prefill_gemm_kernel (down)")) != MOE_OK) return st;
  }
  return MOE_OK;
}

// The A-quantised mode on the block-scaled FP4 MMA: x and h quantised to MXFP4
// (OCP MX), codes and E8M0 scales straight into kind::mxf4.  Buffers: b.xg holds
// the packed x codes [P][H/2], b.xg16 their scales [P][H/32], b.hs the packed h
// codes [P][I/2] followed (256-aligned) by their scales [P][I/32].
static int sm_count_prefill() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

moe_status grouped_gemm_mxf4(const moe_expert_views* v, const uint16_t* x, int T, int k, const int32_t* slots,
                             const GgBufs& b, int32_t* d_error, cudaStream_t stream) {
  const int H = v->H, I = v->I, S = v->fp4_num_slots;
  const size_t P = (size_t)T * k;
  moe_status st = group_pairs_multi(slots, (int)P, S, b.offsets, b.perm, d_error, b.cnt, stream);
  if (st != MOE_OK) return st;
  prefill_items_kernel<<<1, 1024, 0, stream>>>(b.offsets, S, kMxNMax, b.items, b.nitems);
  if ((st = check_launch("prefill_items_kernel")) != MOE_OK) return st;
  uint8_t* xq = reinterpret_cast<uint8_t*>(b.xg);
  uint8_t* xsc = reinterpret_cast<uint8_t*>(b.xg16);
  uint8_t* hq = reinterpret_cast<uint8_t*>(b.hs);
  uint8_t* hsc = hq + a256(P * (size_t)I / 2);
  {
    const int blocks = (int)std::min<size_t>((P + 7) / 8, 152 * 16);
    gather_mxq_kernel<<<blocks, 256, 0, stream>>>(x, H, k, b.perm, b.offsets, S, xq, xsc);
    if ((st = check_launch("gather_mxq_kernel")) != MOE_OK) return st;
  }
  const size_t B = fp4_bytes(H, I);
  const uint8_t* pool = v->fp4_slots;
  const size_t hi = (size_t)H * I;
  const uint8_t* w1c = pool;
  const uint8_t* w1s = pool + hi / 2;
  const uint8_t* w3c = pool + (hi / 2 + hi / 32);
  const uint8_t* w3s = w3c + hi / 2;
  const uint8_t* w2c = pool + 2 * (hi / 2 + hi / 32);
  const uint8_t* w2s = w2c + hi / 2;
  CUtensorMap m1, m3, m2, mx, mh;
  if ((st = map_codes_sw128(&m1, w1c, H / 2, I, S, B, 128)) != MOE_OK) return st;
  if ((st = map_codes_sw128(&m3, w3c, H / 2, I, S, B, 128)) != MOE_OK) return st;
  if ((st = map_codes_sw128(&m2, w2c, I / 2, H, S, B, 128)) != MOE_OK) return st;
  if ((st = map_codes_sw128(&mx, xq, H / 2, P, 0, 0, 64)) != MOE_OK) return st;
  if ((st = map_codes_sw128(&mh, hq, I / 2, P, 0, 0, 64)) != MOE_OK) return st;
  {
    cudaError_t e = cudaFuncSetAttribute(mxf4_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMxSmem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(mxf4_gemm_kernel)");
  }
  const int max_items = (int)std::min<size_t>((size_t)S, P) + (int)(P / kMxNMax) + 1;
  MxArgs ma{};
  ma.H = H;
  ma.I = I;
  ma.S = S;
  ma.P = (int)P;
  ma.B = B;
  ma.items = b.items;
  ma.n_items = b.nitems;
  ma.max_items = max_items;
  ma.perm = b.perm;
  ma.hq = hq;
  ma.hsc = hsc;
  ma.o = b.o;
  ma.err = d_error;
  // GEMM1: gate/up over K = H, 128 features (their w1 and w3 rows) per CTA
  ma.mode = 0;
  ma.K = H;
  ma.tiles = I / 128;
  ma.sc0 = w1s;
  ma.sc1 = w3s;
  ma.bsc = xsc;
  ma.ctr = b.nitems + 1;
  // persistent: one CTA per SM (its tensor memory is the SM's 512 columns)
  const int grid = (int)std::min<long long>(sm_count_prefill(), (long long)max_items * (I / 128));
  {
    ProfScope ps(MOE_K_GEMM_GATEUP, stream);
    cudaError_t le = launch_pdl(mxf4_gemm_kernel, dim3(grid), dim3(kMxThreads), (size_t)kMxSmem, stream, m1, m3, mx, ma);
    if (le != cudaSuccess) return cuda_fail(le, "mxf4_gemm_kernel (gate/up)");
  }
  if ((st = check_launch("mxf4_gemm_kernel (gate/up)")) != MOE_OK) return st;
  // GEMM2: down over K = I, 256 output features per CTA
  ma.mode = 1;
  ma.K = I;
  ma.tiles = H / 256;
  ma.sc0 = w2s;
  ma.sc1 = w2s;
  ma.bsc = hsc;
  ma.ctr = b.nitems + 2;
  {
    ProfScope ps(MOE_K_GEMM_DOWN, stream);
    cudaError_t le = launch_pdl(mxf4_gemm_kernel, dim3(grid), dim3(kMxThreads), (size_t)kMxSmem, stream, m2, m2, mh, ma);
    if (le != cudaSuccess) return cuda_fail(le, "mxf4_gemm_kernel (down)");
  }
  return check_launch("mxf4_gemm_kernel (down)");
}

// rank-2 byte map: (x: row bytes, y: rows)
static moe_status map_bytes2(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_x,
                             uint32_t box_y) {
  auto fn = tensor_map_encoder();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_x, box_y};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (shared weights) failed: %d", (int)r);
  return MOE_OK;
}

moe_status grouped_gemm_shared_fp8(const moe_expert_views* v, const __half* xs, const int* xsig, int T,
                                   __nv_bfloat16* hs, float* o, int o_row0, int32_t* d_error,
                                   cudaStream_t stream) {
  using C = PfShared;
  const int H = v->H, I = v->I;
  // FP8 expert layout: w1 codes [I, H] + fp32 row scales [I], w3 likewise, w2 codes [H, I] + scales [H]
  const size_t hi = (size_t)H * I;
  const uint8_t* w1 = v->shared;
  const uint8_t* w3 = w1 + hi + (size_t)I * 4;
  const uint8_t* w2 = w3 + hi + (size_t)I * 4;
  CUtensorMap m1, m3, m2, mx16, mh;
  moe_status st;
  if ((st = map_bytes2(&m1, w1, H, I, 64, 128)) != MOE_OK) return st;
  if ((st = map_bytes2(&m3, w3, H, I, 64, 128)) != MOE_OK) return st;
  if ((st = map_bytes2(&m2, w2, I, H, 64, 256)) != MOE_OK) return st;
  if ((st = map_bf16_rows(&mx16, xs, H, T, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)) != MOE_OK) return st;
  if ((st = map_bf16_rows(&mh, hs, I, T)) != MOE_OK) return st;
  {
    cudaError_t e = cudaFuncSetAttribute(prefill_gemm_kernel<C, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prefill_gemm_kernel, FP8)");
  }
  const int items = (T + C::kNMax - 1) / C::kNMax;
  PfArgs pa{};
  pa.H = H;
  pa.I = I;
  pa.k = 1;
  pa.S = 1;
  pa.xsig = xsig;
  pa.hs = hs;
  pa.o = o;
  pa.err = d_error;
  pa.rows = T;
  pa.o_row0 = o_row0;
  // gate/up: 128 features (their w1 and w3 rows) per CTA
  pa.mode = 0;
  pa.K = H;
  pa.tiles = I / 128;
  pa.rs0 = reinterpret_cast<const float*>(w1 + hi);
  pa.rs1 = reinterpret_cast<const float*>(w3 + hi);
  {
    ProfScope ps(MOE_K_GATEUP, stream);
    prefill_gemm_kernel<C, true><<<items * pa.tiles, kPfThreads, C::kSmem, stream>>>(m1, m3, mx16, mx16, pa);
  }
  if ((st = check_launch("prefill_gemm_kernel (shared gate/up)")) != MOE_OK) return st;
  // down: 256 output features per CTA
  pa.mode = 1;
  pa.K = I;
  pa.tiles = H / 256;
  pa.rs0 = reinterpret_cast<const float*>(w2 + hi);
  pa.rs1 = pa.rs0;
  {
    ProfScope ps(MOE_K_DOWN, stream);
    prefill_gemm_kernel<C, true><<<items * pa.tiles, kPfThreads, C::kSmem, stream>>>(m2, m2, mh, mh, pa);
  }
  return check_launch("prefill_gemm_kernel (shared down)");
}

struct PfLayout {
  size_t index, xg, xg16, hs, o, total;
};

static PfLayout pf_layout(int H, int I, int T, int k, int S) {
  const size_t P = (size_t)T * k;
  PfLayout L;
  size_t off = 0;
  L.index = off;
  off = a256(off + gg_index_bytes(T, k, S));
  L.xg = off;
  off = a256(off + P * H * 2);
  L.xg16 = off;
  off = a256(off + P * H * 2);
  L.hs = off;
  off = a256(off + P * I * 2);
  L.o = off;
  off = a256(off + P * H * 4);
  L.total = off;
  return L;
}

size_t prefill_workspace(int H, int I, int T, int k, int S) { return pf_layout(H, I, T, k, S).total; }

moe_status prefill_forward(const moe_expert_views* v, const uint16_t* x, int T, int k, const int32_t* slots,
                           const float* w, uint16_t* y, void* workspace, size_t ws_bytes, int32_t* d_error,
                           cudaStream_t stream, int prec_mode) {
  const int H = v->H, I = v->I, S = v->fp4_num_slots;
  MOE_ARG(v->fp4_slots && S >= 1, "the grouped GEMM path needs the FP4 pool");
  MOE_ARG(v->int2_slots == nullptr && v->shared == nullptr,
          "the grouped GEMM path takes the FP4 pool only (no 2-bit pool, no shared expert)");
  MOE_ARG(H % 512 == 0 && I % 512 == 0,
          "the grouped GEMM path needs H and I multiples of 512 (16-byte rows of E8M0 scales)");
  MOE_ARG(S <= 16384, "too many slots");
  MOE_ARG(d_error != nullptr, "the grouped GEMM path needs d_error");
  const PfLayout L = pf_layout(H, I, T, k, S);
  MOE_ARG(ws_bytes >= L.total, "workspace too small: %zu < %zu", ws_bytes, L.total);
  uint8_t* base = (uint8_t*)workspace;
  GgBufs b;
  gg_carve_index(base + L.index, T, k, S, &b);
  b.xg = (uint16_t*)(base + L.xg);
  b.xg16 = (__half*)(base + L.xg16);
  b.hs = (__nv_bfloat16*)(base + L.hs);
  b.o = (float*)(base + L.o);
  MOE_CUDA(cudaMemsetAsync(d_error, 0, sizeof(int32_t), stream));
  moe_status st = prec_mode == MOE_PREC_A_MXFP4 ? grouped_gemm_mxf4(v, x, T, k, slots, b, d_error, stream)
                                                : grouped_gemm_fp4(v, x, T, k, slots, b, d_error, stream);
  if (st != MOE_OK) return st;
  {
    ProfScope ps(MOE_K_COMBINE, stream);
    dim3 cg((H / 4 + 255) / 256, T);
    prefill_combine_kernel<<<cg, 256, 0, stream>>>(b.o, slots, w, T, k, H, S, y);
  }
  return check_launch("prefill_combine_kernel");
}

}  // namespace moe

namespace moe {
// Back-to-back kind::mxf4 MMAs (M = 128, N = 256, K = 64) from shared memory,
// one CTA per SM, `iters` groups of four per CTA into one accumulator: the
// block-scaled FP4 tensor rate this GPU sustains with no data movement.
// Operands are E2M1 1.0 codes with unit scales; the one wait is bounded.
__global__ void __launch_bounds__(128, 1) fp4_peak_kernel(int iters, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* A = sm;                // 128 rows x 128 bytes
  uint8_t* Bm = sm + 128 * 128;   // 256 rows x 128 bytes
  uint64_t* bar = (uint64_t*)(Bm + 256 * 128);
  uint32_t* tslot = (uint32_t*)(bar + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < (128 + 256) * 128 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sm)[i] = make_uint4(0x22222222u, 0x22222222u, 0x22222222u, 0x22222222u);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tslot)), "r"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  // unit scales (127) in the scale columns 256 .. 279 of every lane
  {
    const uint32_t u = 0x7f7f7f7fu;
    const uint32_t v[8] = {u, u, u, u, u, u, u, u};
    const uint32_t col = tmem + ((uint32_t)(32 * warp) << 16) + 256;
    tmem_st8(col, v);
    tmem_st8(col + 8, v);
    tmem_st8(col + 16, v);
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    const uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(256 >> 3) << 17) | (1u << 23) |
                           ((uint32_t)(128 >> 4) << 24);
    const uint32_t id2 = idesc | (2u << 4) | (2u << 29);
    const uint64_t ad = umma_desc_sw128(su32(A)), bd = umma_desc_sw128(su32(Bm));
    const uint32_t sf = tmem + 256;
    for (int i = 0; i < iters; ++i) {
      // four K = 64 MMAs into one accumulator (a K = 256 stage), no commit: the
      // issue queue applies back-pressure
      asm volatile(
          "{\n\t.reg .pred e, t;\n\t.reg .b64 a, bb;\n\t.reg .b32 sb;\n\t"
          "elect.sync _|e, 0xffffffff;\n\tsetp.eq.b32 t, 0, 0;\n\tadd.u32 sb, %4, 16;\n\t"
          "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.block32 [%0], %1, %2, %5, [%4], [sb], t;\n\t"
          "add.s64 a, %1, 2;\n\tadd.s64 bb, %2, 2;\n\t"
          "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.block32 [%0], a, bb, %3, [%4], [sb], t;\n\t"
          "add.s64 a, %1, 4;\n\tadd.s64 bb, %2, 4;\n\t"
          "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.block32 [%0], a, bb, %5, [%4], [sb], t;\n\t"
          "add.s64 a, %1, 6;\n\tadd.s64 bb, %2, 6;\n\t"
          "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.block32 [%0], a, bb, %3, [%4], [sb], t;\n\t}" ::"r"(tmem),
          "l"(ad), "l"(bd), "r"(id2), "r"(sf), "r"(idesc)
          : "memory");
    }
    mma_commit_elect(bar);
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, 0, err));
    (void)ok;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
  }
  (void)lane;
}
}  // namespace moe

extern "C" moe_status moe_fp4_mma_peak(int iters, double* tflops, cudaStream_t stream) {
  moe::clear_error();
  MOE_ARG(iters >= 64 && iters % 64 == 0 && tflops, "need iters a positive multiple of 64 and tflops non-null");
  int dev = 0, sms = 0;
  MOE_CUDA(cudaGetDevice(&dev));
  MOE_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const size_t smem = (128 + 256) * 128 + 64 + 1024;
  MOE_CUDA(cudaFuncSetAttribute(moe::fp4_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  int* err = nullptr;
  MOE_CUDA(cudaMallocAsync((void**)&err, sizeof(int), stream));
  MOE_CUDA(cudaMemsetAsync(err, 0, sizeof(int), stream));
  cudaEvent_t e0, e1;
  MOE_CUDA(cudaEventCreate(&e0));
  MOE_CUDA(cudaEventCreate(&e1));
  moe::fp4_peak_kernel<<<sms, 128, smem, stream>>>(iters / 8, err);  // warm-up
  MOE_CUDA(cudaEventRecord(e0, stream));
  moe::fp4_peak_kernel<<<sms, 128, smem, stream>>>(iters, err);
  MOE_CUDA(cudaEventRecord(e1, stream));
  moe_status st = moe::check_launch("fp4_peak_kernel");
  int h_err = 0;
  if (st == MOE_OK) {
    cudaError_t e = cudaEventSynchronize(e1);
    if (e != cudaSuccess) st = moe::cuda_fail(e, "cudaEventSynchronize");
  }
  float ms = 0.f;
  if (st == MOE_OK) cudaEventElapsedTime(&ms, e0, e1);
  if (st == MOE_OK) cudaMemcpy(&h_err, err, sizeof(int), cudaMemcpyDeviceToHost);
  cudaFreeAsync(err, stream);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (st != MOE_OK) return st;
  if (h_err) return moe::fail(MOE_ERR_TIMEOUT, "fp4 peak probe: a commit wait gave up");
  // 4 MMAs of 2 * 128 * 256 * 64 flops per iteration and CTA
  *tflops = (double)sms * iters * 4.0 * 2.0 * 128 * 256 * 64 / (ms * 1e-3) / 1e12;
  return MOE_OK;
}

extern "C" size_t moe_expert_prefill_workspace(const moe_expert_views* v, int T, int k) {
  if (!v || T < 0 || k < 1) return 0;
  return moe::prefill_workspace(v->H, v->I, T, k, v->fp4_num_slots);
}

extern "C" moe_status moe_expert_prefill_prec(const moe_expert_views* v, const uint16_t* x, int T, int k,
                                              const int32_t* slots, const float* w, int prec_mode, uint16_t* y,
                                              void* workspace, size_t workspace_bytes, int32_t* d_error,
                                              cudaStream_t stream) {
  moe::clear_error();
  MOE_ARG(v != nullptr, "views is null");
  MOE_ARG(T >= 0 && k >= 1 && k <= 64, "need T >= 0 and 1 <= k <= 64");
  MOE_ARG(prec_mode == MOE_PREC_W4A16 || prec_mode == MOE_PREC_A_MXFP4, "unknown precision mode %d", prec_mode);
  if (T == 0) return MOE_OK;
  MOE_ARG(x && slots && w && y && workspace, "null pointer");
  MOE_ARG(((uintptr_t)workspace & 255) == 0, "workspace must be 256-byte aligned");
  MOE_ARG(((uintptr_t)x & 15) == 0, "x must be 16-byte aligned");
  return moe::prefill_forward(v, x, T, k, slots, w, y, workspace, workspace_bytes, d_error, stream, prec_mode);
}

extern "C" moe_status moe_expert_prefill(const moe_expert_views* v, const uint16_t* x, int T, int k,
                                         const int32_t* slots, const float* w, uint16_t* y, void* workspace,
                                         size_t workspace_bytes, int32_t* d_error, cudaStream_t stream) {
  return moe_expert_prefill_prec(v, x, T, k, slots, w, MOE_PREC_W4A16, y, workspace, workspace_bytes, d_error,
                                 stream);
}

namespace moe {
// One thread per 32-element block: its 16 code bytes and its scale byte.
__global__ void mx_quantize_kernel(const uint16_t* x, long long blocks, uint8_t* codes, uint8_t* scales) {
  for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < blocks;
       b += (long long)gridDim.x * blockDim.x) {
    float f[32];
    const uint4* src = reinterpret_cast<const uint4*>(x + b * 32);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint4 v = src[u];
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        f[8 * u + 2 * q] = __uint_as_float(w4[q] << 16);
        f[8 * u + 2 * q + 1] = __uint_as_float(w4[q] & 0xffff0000u);
      }
    }
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) am = fmaxf(am, fabsf(f[i]));
    const uint32_t sb = mx_scale_byte(am);
    const float inv = mx_inv_scale(sb);
    uint32_t o[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t word = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) word |= mx_code(f[8 * w + i], inv) << (4 * i);
      o[w] = word;
    }
    reinterpret_cast<uint4*>(codes)[b] = make_uint4(o[0], o[1], o[2], o[3]);
    scales[b] = (uint8_t)sb;
  }
}
}  // namespace moe

extern "C" moe_status moe_mx_quantize(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* scales,
                                      cudaStream_t stream) {
  moe::clear_error();
  MOE_ARG(rows >= 0 && K >= 0 && K % 32 == 0, "need rows >= 0 and K a multiple of 32");
  if (rows == 0 || K == 0) return MOE_OK;
  MOE_ARG(x && codes && scales, "null pointer");
  MOE_ARG(((uintptr_t)x & 15) == 0 && ((uintptr_t)codes & 15) == 0, "x and codes must be 16-byte aligned");
  const long long blocks = (long long)rows * (K / 32);
  const int grid = (int)std::min<long long>((blocks + 255) / 256, 152LL * 8);
  moe::mx_quantize_kernel<<<grid, 256, 0, stream>>>(x, blocks, codes, scales);
  return moe::check_launch("mx_quantize_kernel");
}
