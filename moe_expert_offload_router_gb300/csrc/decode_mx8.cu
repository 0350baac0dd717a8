// Block-scaled tensor-core GEMMs of the decode forward: the grouped expert
// MLP of decode batches (up to 64 tokens per expert) on
// tcgen05.mma.kind::mxf8f6f4 with no weight conversion at all.
//
// "Running DeepSeek-V4-Flash across four free GPUs", section "What the expert
// cache actually does" (the grouped expert GEMM over the slot views); "An
// elephant through a straw", section "Rig, model & methodology" (MXFP4
// experts: E2M1 codes with one E8M0 scale per 32 weights; one FP8 shared
// expert).
//
// The A operand is the expert's weight rows as stored in the slot pool: TMA
// copies the packed E2M1 codes with the 16U4_ALIGN16B element type, which
// lays 16 codes into each 16-byte unit of shared memory (8 bytes of codes, 8
// bytes of gap), the operand layout the tensor core reads E2M1 from, and the
// rows' E8M0 block scales go to tensor memory as the MMA's A scale factors.
// The FP8 shared expert's E4M3 rows load as bytes with a unit A scale; its
// per-row fp32 scales multiply the accumulators.  The B operand is the
// activations, each 32-element block along K scaled by a power of two and
// carried as two E4M3 terms hi + lo (mx.cuh); a bf16 input is held exactly in
// all but subnormal-lo cases, so the products are those of the bf16 path.
// Groups hold up to 48 tokens; the hi and lo rows of a stage stack into one
// B operand of 2n rows (one MMA per K slice and tile), and the epilogue adds
// the accumulator's two halves.
//
// Persistent CTAs, two per SM (192 threads, 98 KB of shared memory and 256
// tensor-memory columns each): one CTA's TMA engine moves the 64-byte rows of
// the packed E2M1 tiles at about two thirds of an SM's share of HBM, two
// together at the full rate, and one CTA streams while the other runs its
// epilogue.  Items = (token group, feature tile): CTA c starts with item c and
// draws the next from a global counter, published to the other warps through
// a small queue in shared memory (the tail is at most about one item):
//   warp 0      TMA: two 128-row A tiles and the group's hi/lo rows per
//               128-element K stage, two stages deep; draws the items and
//               prefetches each next item's A scale rows into L2
//   warp 1      TMEM allocation; MMA issue (one elected lane, one asm block
//               per stage), commits to the stage's "empty" barrier and, after
//               the item's last stage, to the accumulators' "full" barrier
//   warps 2-5   per item: the A and B scale words of every stage into their
//               TMEM lane quadrant (A rows read 16 bytes per four stages, the
//               group's B scale rows copied to shared memory once, one item
//               ahead), then the
//               epilogue: gate/up -> h = SiLU(gate) * up, itself split into
//               E4M3 hi/lo with a scale per 32 features (the down GEMM's B
//               operand, in the same sorted row order); down -> fp32 rows of
//               o per pair for the router-weighted combine
// Launched with programmatic stream serialization: barriers, tensor memory and
// tensor-map prefetches are set up while the previous kernel finishes.  Every
// mbarrier wait gives up after one second and records MOE_ERR_TIMEOUT.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "grouped_gemm.cuh"
#include "mx.cuh"
#include "tcgen05.cuh"

namespace moe {

constexpr int kM8Threads = 192;                 // 6 warps: TMA, MMA, four scale-factor / epilogue warps
constexpr int kM8CtasPerSm = 2;                 // two CTAs stream each SM's share of HBM
constexpr int kM8Stages = 2;
constexpr int kM8KStage = 128;                  // K elements per stage: one 128-byte swizzled row
constexpr int kM8ATile = 128 * 128;             // one 128-row A tile of a stage in shared memory
constexpr int kM8BBytes = 2 * kMx8MaxRows * 128;  // hi rows, then lo rows
constexpr int kM8Stage = 2 * kM8ATile + kM8BBytes;
constexpr int kM8OffBar = kM8Stages * kM8Stage;
constexpr int kM8OffSB = kM8OffBar + 256;       // the group's B scale rows, padded by 16 bytes
constexpr int kM8SBBytes = kMx8MaxRows * (4096 / 32 + 16);  // K up to 4096
constexpr int kM8Smem = kM8OffSB + 2 * kM8SBBytes + 1024;  // two B scale buffers (this item, the next)
constexpr int kM8AccCols = 2 * kMx8MaxRows;     // TMEM columns per accumulator (hi and lo halves)
constexpr int kM8SfBase = 2 * kM8AccCols;       // the two accumulators, then the scale factors
constexpr int kM8SfCols = 16;                   // per stage: A tile 0 +0..3, A tile 1 +4..7, B +8..10
constexpr int kM8TmemCols = 256;                // half of an SM's tensor memory
static_assert(kM8SfBase + kM8Stages * kM8SfCols <= kM8TmemCols, "tensor memory columns");
static_assert(kM8CtasPerSm * (kM8Smem + 1024) <= 228 * 1024, "shared memory of two CTAs per SM");
static_assert(kM8AccCols % 32 == 0 && kM8AccCols <= 96, "accumulator width (three B scale columns)");
constexpr int kM8Queue = 4;                     // items published ahead to the consumer warps
static_assert((2 * kM8Stages + 4 + 2 * kM8Queue) * 8 + 8 + 4 * kM8Queue <= 256, "barrier area");

struct Mx8Args {
  int mode;          // 0: gate/up + SwiGLU -> h hi/lo; 1: down -> o
  int K;             // H (mode 0) or I (mode 1)
  int H, I, T, P;
  int tiles;         // feature tiles per group: I / 128 (mode 0) or H / 256 (mode 1)
  int max_groups;    // capacity of the group list
  const uint8_t* fp4;
  int n4;
  size_t b4;         // bytes per FP4 expert
  size_t sc0, sc1;   // byte offsets of the A tiles' E8M0 scales in an expert (mode 0: w1, w3; mode 1: w2)
  const uint8_t* shared;
  const float* rs0;  // shared expert row scales: w1 (mode 0) or w2 (mode 1)
  const float* rs1;  // w3 (mode 0)
  const uint8_t* bsc;  // B scale bytes [P + T][K / 32]
  const int* hdr;      // [0] groups, [1] routed groups (the shared expert's follow)
  int* ctr;            // item counter (zeroed by the plan): items past the first gridDim.x are drawn from it
  const Group* groups;
  const int* perm;     // sorted position -> pair index
  uint8_t* hhi;        // mode 0 out: [P + T][I] E4M3 hi, lo, and scale bytes [P + T][I / 32]
  uint8_t* hlo;
  uint8_t* hsc;
  float* o;            // mode 1 out: [P + T][H] (row = pair index, or P + token for the shared expert)
  int* err;
};

struct M8Item {
  bool run;          // a group this kernel computes
  bool fp8;          // the shared expert
  int slot, begin, count, brow0, f0, n16;
};

// Item it of the list: groups in the order shared expert first, then routed;
// tile fastest.  2-bit groups belong to the CUDA-core kernels and are skipped;
// a group the plan never produces is skipped and flagged (by warp 1 only).
__device__ __forceinline__ M8Item m8_item(const Mx8Args& a, int it, int ng, int nr, bool flag) {
  M8Item r;
  r.run = false;
  const int gi = it / a.tiles, tile = it % a.tiles;
  const Group g = a.groups[(nr + gi) % ng];
  r.fp8 = g.pool == MOE_POOL_SHARED;
  r.slot = g.slot;
  r.begin = g.begin;
  r.count = g.count;
  r.f0 = a.mode == 0 ? tile * 128 : tile * 256;
  r.n16 = (g.count + 15) & ~15;
  if (g.pool == MOE_POOL_INT2) return r;
  bool ok = g.count >= 1 && g.count <= kMx8MaxRows && g.begin >= 0;
  if (r.fp8) {
    ok = ok && a.shared != nullptr && g.begin + g.count <= a.T;
    r.brow0 = a.P + g.begin;
  } else {
    ok = ok && g.pool == MOE_POOL_FP4 && g.slot >= 0 && g.slot < a.n4 && g.begin + g.count <= a.P;
    r.brow0 = g.begin;
  }
  if (!ok) {
    if (flag) atomicCAS(a.err, 0, MOE_ERR_INVALID);
    return r;
  }
  r.run = true;
  return r;
}

// Four K = 32 slices of one stage for both accumulators, from one elected
// lane: one MMA per slice and tile, B = the stage's hi rows then its lo rows
// (N = 2 n).  Slice j advances the descriptors 32 bytes and selects byte j of
// the scale-factor words (the A and B scale-factor IDs of the instruction
// descriptor).
__device__ __forceinline__ void m8_stage(uint32_t d0, uint32_t d1, uint64_t a0, uint64_t a1, uint64_t b,
                                         uint32_t idesc, uint32_t sfa0, uint32_t sfa1, uint32_t sfb, uint32_t acc,
                                         uint64_t* bar) {
#define M8_MMA(D, A, SFA, P) \
  "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.block32 [" D "], " A ", bb, id, [" SFA "], [%8], " P ";\n\t"
#define M8_SLICE(OFF, IDOFF, P)                                                                             \
  "add.s64 a, %2, " OFF ";\n\tadd.s64 c, %3, " OFF ";\n\tadd.s64 bb, %4, " OFF ";\n\tadd.u32 id, %5, " IDOFF \
  ";\n\t" M8_MMA("%0", "a", "%6", P) M8_MMA("%1", "c", "%7", P)
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t.reg .b64 a, c, bb;\n\t.reg .b32 id;\n\t"
      "elect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %9, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t" M8_SLICE("0", "0", "p")
          M8_SLICE("2", "536870928", "t") M8_SLICE("4", "1073741856", "t") M8_SLICE("6", "1610612784", "t")
              "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%10];\n\t}" ::"r"(d0),
      "r"(d1), "l"(a0), "l"(a1), "l"(b), "r"(idesc), "r"(sfa0), "r"(sfa1), "r"(sfb), "r"(acc), "r"(su32(bar))
      : "memory");
#undef M8_SLICE
#undef M8_MMA
}
// The immediates above are j * (2^29 + 2^4) for j = 1, 2, 3: the A scale-factor
// ID (bits 29-30) and the B scale-factor ID (bits 4-5) both set to j.
static_assert(536870928u == (1u << 29) + (1u << 4) && 1610612784u == 3u * ((1u << 29) + (1u << 4)),
              "scale-factor ID immediates");

__device__ __forceinline__ uint4 ldg_u128(const uint8_t* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }


// L2 prefetch of an FP4 item's A scale rows (two runs of 128 rows x K / 32
// bytes, contiguous in the expert), so the scale-factor warps' loads hit L2.
__device__ __forceinline__ void m8_prefetch_scales(const Mx8Args& a, const M8Item& m) {
  if (!m.run || m.fp8) return;
  const uint32_t sbytes = (uint32_t)a.K / 32;
  const uint8_t* e = a.fp4 + (size_t)m.slot * a.b4;
  const int row1 = a.mode == 0 ? m.f0 : m.f0 + 128;
  const uint8_t* p0 = e + a.sc0 + (size_t)m.f0 * sbytes;
  const uint8_t* p1 = e + a.sc1 + (size_t)row1 * sbytes;
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p0), "r"(128u * sbytes) : "memory");
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p1), "r"(128u * sbytes) : "memory");
}

__global__ void __launch_bounds__(kM8Threads, kM8CtasPerSm)
    mx8_gemm_kernel(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
                    const __grid_constant__ CUtensorMap mS0, const __grid_constant__ CUtensorMap mS1,
                    const __grid_constant__ CUtensorMap mBh, const __grid_constant__ CUtensorMap mBl, Mx8Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full = (uint64_t*)(sm + kM8OffBar);  // [kM8Stages]: TMA bytes + the four scale-factor warps
  uint64_t* empty = full + kM8Stages;             // [kM8Stages]: the stage's MMAs completed
  uint64_t* accf = empty + kM8Stages;             // the item's MMAs completed
  uint64_t* acce = accf + 1;                      // the epilogue has read the accumulators
  uint64_t* drain = acce + 1;
  uint64_t* qfull = drain + 1;                    // [kM8Queue]: an item index published
  uint64_t* qempty = qfull + kM8Queue;            // [kM8Queue]: the five consumer warps have read it
  uint64_t* sbar = qempty + kM8Queue;             // the four scale-factor warps (copy of the B scale rows)
  uint32_t* tmem_slot = (uint32_t*)(sbar + 1);
  volatile int* itq = (volatile int*)(tmem_slot + 1);  // [kM8Queue] item indices, -1 = no more
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = a.K / kM8KStage;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (const CUtensorMap* m : {&mA0, &mA1, &mS0, &mS1, &mBh, &mBl})
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
  }
  // the barriers and the tensor memory above do not depend on the previous
  // kernel (the plan, or the gate/up GEMM): set them up before waiting for it
  int ng = 0, nr = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kM8Stages; ++s) {
      mbar_init(&full[s], 1 + 4);  // the TMA thread's expect_tx arrival + the scale-factor warps
      mbar_init(&empty[s], 1);
    }
    mbar_init(accf, 1);
    mbar_init(acce, 4);
    mbar_init(drain, 1);
    for (int j = 0; j < kM8Queue; ++j) {
      mbar_init(&qfull[j], 1);
      mbar_init(&qempty[j], 1 + 4);  // the MMA warp and the four scale-factor / epilogue warps
    }
    mbar_init(sbar, 4);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(kM8TmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  ng = a.hdr[0];
  nr = a.hdr[1];
  if (ng < 0 || ng > a.max_groups || nr < 0 || nr > ng) {
    if (threadIdx.x == 0) atomicCAS(a.err, 0, MOE_ERR_INVALID);
    ng = 0;
  }
  const int n_items = ng * a.tiles;
  // q-th item of this CTA for a consumer warp (whole warp): false on timeout
  auto next_item = [&](uint32_t q, int& it) -> bool {
    const int j = q % kM8Queue;
    if (!__all_sync(0xffffffffu, mbar_wait_fast(&qfull[j], (q / kM8Queue) & 1, a.err))) return false;
    it = itq[j];
    __syncwarp();
    if (lane == 0) mbar_arrive(&qempty[j]);
    return true;
  };

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      uint32_t gs = 0, q = 0;
      auto publish = [&](int it) -> bool {
        const int j = q % kM8Queue;
        const uint32_t r = q / kM8Queue;
        if (r > 0 && !mbar_wait_fast(&qempty[j], (r - 1) & 1, a.err)) return false;
        itq[j] = it;
        mbar_arrive(&qfull[j]);  // release: the index is visible to the warps that wait on it
        ++q;
        return true;
      };
      int cur = (int)blockIdx.x < n_items ? (int)blockIdx.x : -1;
      ok = publish(cur);
      if (cur >= 0) m8_prefetch_scales(a, m8_item(a, cur, ng, nr, false));
      while (ok && cur >= 0) {
        // the next item's ticket: its latency overlaps this item's loads
        const int ticket = atomicAdd(a.ctr, 1);
        const M8Item m = m8_item(a, cur, ng, nr, false);
        if (m.run) {
          const int nbx = m.n16 / 16;
          const uint32_t bytes = (m.fp8 ? 2u * kM8ATile : (uint32_t)kM8ATile) + 2u * (uint32_t)nbx * 2048u;
          const int row1 = a.mode == 0 ? m.f0 : m.f0 + 128;
          for (int ks = 0; ks < nk; ++ks, ++gs) {
            const int s = gs % kM8Stages;
            const uint32_t r = gs / kM8Stages;
            if (r > 0 && !(ok = mbar_wait_fast(&empty[s], (r - 1) & 1, a.err))) break;
            uint8_t* st = sm + s * kM8Stage;
            mbar_expect_tx(&full[s], bytes);
            const int x = ks * kM8KStage;  // element coordinate: 64 (FP4) or 128 (E4M3) bytes, 16-byte multiples
            if (m.fp8) {
              tma_2d(st, &mS0, x, m.f0, &full[s]);
              tma_2d(st + kM8ATile, &mS1, x, row1, &full[s]);
            } else {
              tma_3d(st, &mA0, x, m.f0, m.slot, &full[s]);
              tma_3d(st + kM8ATile, &mA1, x, row1, m.slot, &full[s]);
            }
            uint8_t* bd = st + 2 * kM8ATile;
            for (int bx = 0; bx < nbx; ++bx) {
              tma_2d(bd + bx * 2048, &mBh, x, m.brow0 + 16 * bx, &full[s]);
              tma_2d(bd + (nbx + bx) * 2048, &mBl, x, m.brow0 + 16 * bx, &full[s]);
            }
          }
        }
        if (!ok) break;
        int nxt = ticket + (int)gridDim.x;
        if (nxt >= n_items) nxt = -1;
        if (!(ok = publish(nxt))) break;
        if (nxt >= 0) m8_prefetch_scales(a, m8_item(a, nxt, ng, nr, false));
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
      int it;
      if (!(ok = next_item(qi, it)) || it < 0) break;
      const M8Item m = m8_item(a, it, ng, nr, true);
      if (!m.run) continue;
      // the epilogue of the previous item has read the accumulators
      if (i > 0 && !(ok = __all_sync(0xffffffffu, mbar_wait_fast(acce, (i - 1) & 1, a.err)))) break;
      ++i;
      tc_fence_after();
      // E2M1 (5) or E4M3 (0) A, E4M3 B, fp32 D, K-major both, E8M0 scales, M = 128, N = 2 n16
      const uint32_t idesc = ((m.fp8 ? 0u : 5u) << 7) | ((uint32_t)(2 * m.n16 >> 3) << 17) | (1u << 23) |
                             ((uint32_t)(128 >> 4) << 24);
      const uint32_t d0 = tmem, d1 = tmem + kM8AccCols;
      for (int ks = 0; ks < nk; ++ks, ++gs) {
        const int s = gs % kM8Stages;
        const uint32_t r = gs / kM8Stages;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait_fast(&full[s], r & 1, a.err)))) break;
        tc_fence_after();
        uint8_t* st = sm + s * kM8Stage;
        const uint64_t ad0 = umma_desc_sw128(su32(st)), ad1 = umma_desc_sw128(su32(st + kM8ATile));
        const uint64_t bd = umma_desc_sw128(su32(st + 2 * kM8ATile));
        const uint32_t sf = tmem + kM8SfBase + kM8SfCols * s;
        m8_stage(d0, d1, ad0, ad1, bd, idesc, sf, sf + 4, sf + 8, ks != 0, &empty[s]);
      }
      if (ok) mma_commit_elect(accf);
    }
    // every MMA this warp issued has completed before tensor memory is freed
    mma_commit_elect(drain);
    __syncwarp();
    mbar_wait(drain, 0, a.err);
  } else {
    // warps 2-5: lane quadrant q = warp % 4 of tensor memory.  Per item, the
    // scale factors of every stage (A row 32 q + lane of each tile at column
    // +q of its 4-column group; B rows 32 c + lane at column +8 + c), then
    // the epilogue once the item's MMAs have completed.  The scale rows are
    // read whole, once per item: each lane reads its two A rows 16 bytes (four
    // stages) at a time, one group of four ahead, and the group's B rows go to
    // shared memory in one coalesced copy by the four warps; scattered 4-byte
    // loads per stage cost about as many L2 requests as the TMA's own and
    // slowed it down.  The B
    // rows have two buffers: the next item's are copied right after the
    // current item's last scale-factor store, while its last MMAs complete,
    // so the next item's first stage does not wait for the copy.
    const int q = warp & 3;
    const int tid = threadIdx.x - 64;  // 0 .. 127 over the four warps
    const int sbytes = a.K / 32;
    const int srow = sbytes + 16;      // padded row of the B scale copy (4-way bank conflicts at most)
    uint8_t* sB = sm + kM8OffSB;
    bool ok = true;
    uint32_t gs = 0, i = 0, nsync = 0;
    // the four warps meet (an mbarrier with a bounded wait, so a warp that gave
    // up cannot leave the others waiting)
    auto group_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(sbar);
      return __all_sync(0xffffffffu, mbar_wait_fast(sbar, (nsync++) & 1, a.err));
    };
    uint32_t qi = 0;
    // the next item that runs (items no role computes are skipped): its
    // index, -1 at the end of the list, -2 on a timeout
    auto take_run = [&](M8Item& mm) -> int {
      for (;;) {
        int it;
        if (!next_item(qi++, it)) return -2;
        if (it < 0) return -1;
        mm = m8_item(a, it, ng, nr, false);
        if (mm.run) return it;
      }
    };
    // an item's B scale rows (contiguous in global memory) -> shared buffer b
    auto copy_b = [&](const M8Item& mm, int b) {
      uint8_t* dst = sB + b * kM8SBBytes;
      const uint8_t* gB = a.bsc + (size_t)mm.brow0 * sbytes;
      const int cpr = sbytes / 16, n = mm.count * cpr;
      for (int c = tid; c < n; c += 128)
        *reinterpret_cast<uint4*>(dst + (c / cpr) * srow + 16 * (c % cpr)) = ldg_u128(gB + 16 * c);
    };
    // Each copy is followed by a group sync, so every warp's share is in place
    // before any warp reads the buffer; a buffer is copied into again only
    // after every warp has passed the sync that followed the copy after its
    // last reader (the item two back), so no copy overtakes a reader.  The
    // sync sits before the epilogue: a warp goes from its own epilogue
    // straight to the next item's scale factors.
    M8Item m;
    int it = take_run(m);
    ok = it != -2;
    int buf = 0;
    bool have_pre = false;  // pre0 / pre1 hold the item's first 16 scale bytes of each A row
    uint4 pre0 = make_uint4(0, 0, 0, 0), pre1 = pre0;
    if (it >= 0) {
      copy_b(m, 0);
      ok = group_sync();
    }
    while (ok && it >= 0) {
      const uint8_t* sBb = sB + buf * kM8SBBytes;
      const uint8_t* sa0 = nullptr;
      const uint8_t* sa1 = nullptr;
      if (!m.fp8) {
        const uint8_t* e = a.fp4 + (size_t)m.slot * a.b4;
        const int r0 = m.f0 + 32 * q + lane, r1 = (a.mode == 0 ? m.f0 : m.f0 + 128) + 32 * q + lane;
        sa0 = e + a.sc0 + (size_t)r0 * sbytes;
        sa1 = e + a.sc1 + (size_t)r1 * sbytes;
      }
      const uint32_t* sbw[3];  // this lane's B rows in the shared copy
#pragma unroll
      for (int c = 0; c < 3; ++c) {
        int tk = 32 * c + lane;
        if (tk >= m.n16) tk -= m.n16;  // B rows n16 .. 2 n16 - 1 are the lo terms
        if (tk >= m.count) tk = 0;     // columns past the group: any valid row
        sbw[c] = reinterpret_cast<const uint32_t*>(sBb + tk * srow);
      }
      auto store = [&](uint32_t wa0, uint32_t wa1, int ks) -> bool {
        const int s = gs % kM8Stages;
        const uint32_t r = gs / kM8Stages;
        // the slot's previous stage (gs - kM8Stages) must have finished its MMAs
        if (r > 0 && !__all_sync(0xffffffffu, mbar_wait_fast(&empty[s], (r - 1) & 1, a.err))) return false;
        const uint32_t col = tmem + ((uint32_t)(32 * q) << 16) + kM8SfBase + kM8SfCols * s;
        tmem_st1(col + q, wa0);
        tmem_st1(col + 4 + q, wa1);
        tmem_st1(col + 8, sbw[0][ks]);
        tmem_st1(col + 9, sbw[1][ks]);
        tmem_st1(col + 10, sbw[2][ks]);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
        ++gs;
        return true;
      };
      // nk is a multiple of 4 (K a multiple of 512): 16 bytes of an A row hold
      // four stages' words; each group of four is loaded one group ahead
      const uint4 unit = make_uint4(0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu);
      uint4 n0 = m.fp8 ? unit : have_pre ? pre0 : ldg_u128(sa0);
      uint4 n1 = m.fp8 ? unit : have_pre ? pre1 : ldg_u128(sa1);
      for (int ks = 0; ks < nk && ok; ks += 4) {
        const uint4 c0 = n0, c1 = n1;
        if (!m.fp8 && ks + 4 < nk) {
          n0 = ldg_u128(sa0 + 4 * (ks + 4));
          n1 = ldg_u128(sa1 + 4 * (ks + 4));
        }
        if (ok) ok = store(c0.x, c1.x, ks);
        if (ok) ok = store(c0.y, c1.y, ks + 1);
        if (ok) ok = store(c0.z, c1.z, ks + 2);
        if (ok) ok = store(c0.w, c1.w, ks + 3);
      }
      if (!ok) break;
      // the next item's B scale rows go to the other buffer while this item's
      // last MMAs complete
      M8Item mn;
      const int nit = take_run(mn);
      ok = nit != -2;
      if (!ok) break;
      if (nit >= 0) {
        copy_b(mn, buf ^ 1);
        if (!(ok = group_sync())) break;
      }
      // and the first 16 bytes of this lane's two A scale rows (the first
      // four stages' words), so the next item's first stores wait for no load
      uint4 pre0n = make_uint4(0, 0, 0, 0), pre1n = pre0n;
      if (nit >= 0 && !mn.fp8) {
        const uint8_t* e = a.fp4 + (size_t)mn.slot * a.b4;
        const int r0 = mn.f0 + 32 * q + lane, r1 = (a.mode == 0 ? mn.f0 : mn.f0 + 128) + 32 * q + lane;
        pre0n = ldg_u128(e + a.sc0 + (size_t)r0 * sbytes);
        pre1n = ldg_u128(e + a.sc1 + (size_t)r1 * sbytes);
      }

      // epilogue
      if (!(ok = __all_sync(0xffffffffu, mbar_wait_fast(accf, i & 1, a.err)))) break;
      ++i;
      tc_fence_after();
      const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
      const uint32_t lo_off = (uint32_t)m.n16;
      // accumulator columns c0 .. c0 + 15 of tile t: hi half plus lo half
      auto acc16 = [&](int t, int c0, float* v) {
        uint32_t r[16];
        tmem_ld16(tq + (uint32_t)(t * kM8AccCols + c0), r);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
        tmem_ld16(tq + (uint32_t)(t * kM8AccCols + c0) + lo_off, r);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] += __uint_as_float(r[j]);
      };
      if (a.mode == 0) {
        const int f = m.f0 + 32 * q + lane;  // this lane's feature
        const float rg = m.fp8 ? a.rs0[f] : 1.f, ru = m.fp8 ? a.rs1[f] : 1.f;
        uint8_t* hi_base = a.hhi + f;
        uint8_t* lo_base = a.hlo + f;
        uint8_t* sc_base = a.hsc + (m.f0 + 32 * q) / 32;
        for (int c0 = 0; c0 < m.n16; c0 += 16) {
          float g[16], up[16];
          acc16(0, c0, g);
          acc16(1, c0, up);
          float hv[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float hg = 0.5f * (g[j] * rg);
            hv[j] = fmaf(hg, tanh_approx(hg), hg) * (up[j] * ru);
          }
          // a warp's 32 lanes are 32 consecutive features: one scale block of h
          uint32_t sbyte[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const uint32_t am = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(hv[j])));
            sbyte[j] = mx8_scale_byte(__uint_as_float(am));
            hv[j] *= __uint_as_float((254u - sbyte[j]) << 23);
          }
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            uint32_t hi, lo;
            mx8_split2(hv[j], hv[j + 1], hi, lo);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int col = c0 + j + e;
              if (col < m.count) {
                const size_t row = (size_t)(m.brow0 + col);
                hi_base[row * a.I] = (uint8_t)(hi >> (8 * e));
                lo_base[row * a.I] = (uint8_t)(lo >> (8 * e));
                if (lane == 0) sc_base[row * (a.I / 32)] = (uint8_t)sbyte[j + e];
              }
            }
          }
        }
      } else {
        const int fa = m.f0 + 32 * q + lane, fb = fa + 128;
        const float ra = m.fp8 ? a.rs0[fa] : 1.f, rb = m.fp8 ? a.rs0[fb] : 1.f;
        for (int c0 = 0; c0 < m.n16; c0 += 16) {
          float v0[16], v1[16];
          acc16(0, c0, v0);
          acc16(1, c0, v1);
          const int cl = c0 + (lane & 15);
          const int pl = cl < m.count ? (m.fp8 ? a.P + m.begin + cl : a.perm[m.begin + cl]) : 0;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int p = __shfl_sync(0xffffffffu, pl, j);
            if (c0 + j < m.count) {
              float* orow = a.o + (size_t)p * a.H;
              orow[fa] = v0[j] * ra;
              orow[fb] = v1[j] * rb;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce);
      m = mn;
      it = nit;
      buf ^= 1;
      have_pre = nit >= 0 && !mn.fp8;
      pre0 = pre0n;
      pre1 = pre1n;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kM8TmemCols));
  }
}

// ------------------------------------------------------------------- host --

// Packed E2M1 codes of one matrix over every slot: (x: K codes, y: rows,
// z: slots), 16U4_ALIGN16B (16 codes per 16 bytes of shared memory), 128-byte
// swizzle, box of 128 codes by 128 rows (an A tile).
static moe_status map_fp4_rows(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint64_t slots,
                               uint64_t slot_stride) {
  auto fn = tensor_map_encoder();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {K, rows, slots};
  cuuint64_t strides[2] = {K / 2, slot_stride};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (FP4 rows) failed: %d", (int)r);
  return MOE_OK;
}

// Byte rows (E4M3): (x: K bytes, y: rows), 128-byte swizzle, box of 128 bytes by box_rows.
static moe_status map_u8_rows(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows) {
  auto fn = tensor_map_encoder();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[2] = {K, rows};
  cuuint64_t strides[1] = {K};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (E4M3 rows) failed: %d", (int)r);
  return MOE_OK;
}

static int mx8_sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

bool mx8_supported(const moe_expert_views* v) {
  // K stages of 128 elements whose scale words go four stages to a 16-byte
  // load (H, I multiples of 512); the B scale rows' shared copy holds K up to
  // 4096; 256-row down tiles; the 16U4 element type needs 32-byte aligned
  // bases and row strides
  if (v->H % 512 != 0 || v->I % 512 != 0 || v->H > 4096 || v->I > 4096) return false;
  const bool fp4 = v->fp4_slots != nullptr && v->fp4_num_slots > 0;
  if (fp4 && ((uintptr_t)v->fp4_slots & 31) != 0) return false;
  if (v->shared && ((uintptr_t)v->shared & 15) != 0) return false;
  return fp4 || v->shared != nullptr;
}

size_t mx8_bytes(int H, int I, int rows) {
  auto a = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return 2 * a((size_t)rows * H) + a((size_t)rows * H / 32) + 2 * a((size_t)rows * I) + a((size_t)rows * I / 32);
}

void mx8_carve(uint8_t* base, int H, int I, int rows, Mx8Bufs* b) {
  auto a = [](size_t x) { return (x + 255) & ~(size_t)255; };
  size_t off = 0;
  b->xhi = base + off;
  off += a((size_t)rows * H);
  b->xlo = base + off;
  off += a((size_t)rows * H);
  b->xsc = base + off;
  off += a((size_t)rows * H / 32);
  b->hhi = base + off;
  off += a((size_t)rows * I);
  b->hlo = base + off;
  off += a((size_t)rows * I);
  b->hsc = base + off;
}

moe_status mx8_gemm(const moe_expert_views* v, int mode, int T, int k, bool shared, int max_groups, int rows,
                    int* hdr, const Group* groups, const int* perm, const Mx8Bufs& b, float* o,
                    int32_t* d_error, cudaStream_t stream) {
  const int H = v->H, I = v->I, P = T * k;
  const size_t b4 = fp4_bytes(H, I);
  const size_t codes_hi = (size_t)I * H / 2, scales_hi = (size_t)I * H / 32;  // one w1 or w3 matrix
  const size_t off_w3 = codes_hi + scales_hi, off_w2 = 2 * off_w3;
  const size_t f8_mat = (size_t)I * H + (size_t)I * 4;  // one shared w1 or w3 matrix (codes + row scales)
  const uint8_t* sh = shared ? v->shared : nullptr;
  Mx8Args a;
  a.mode = mode;
  a.K = mode == 0 ? H : I;
  a.H = H;
  a.I = I;
  a.T = T;
  a.P = P;
  a.tiles = mode == 0 ? I / 128 : H / 256;
  a.max_groups = max_groups;
  a.fp4 = v->fp4_slots;
  a.n4 = v->fp4_slots ? v->fp4_num_slots : 0;
  a.b4 = b4;
  a.sc0 = mode == 0 ? codes_hi : off_w2 + (size_t)H * I / 2;
  a.sc1 = mode == 0 ? off_w3 + codes_hi : a.sc0;
  a.shared = sh;
  a.rs0 = sh ? reinterpret_cast<const float*>(sh + (mode == 0 ? (size_t)I * H : 2 * f8_mat + (size_t)H * I))
             : nullptr;
  a.rs1 = sh ? reinterpret_cast<const float*>(sh + f8_mat + (size_t)I * H) : nullptr;
  a.bsc = mode == 0 ? b.xsc : b.hsc;
  a.hdr = hdr;
  a.ctr = hdr + 2 + mode;  // zeroed by the plan kernel
  a.groups = groups;
  a.perm = perm;
  a.hhi = b.hhi;
  a.hlo = b.hlo;
  a.hsc = b.hsc;
  a.o = o;
  a.err = d_error;

  CUtensorMap mA0, mA1, mS0, mS1, mBh, mBl;
  moe_status st;
  const int S = a.n4;
  if (a.fp4 && S > 0) {
    if (mode == 0) {
      if ((st = map_fp4_rows(&mA0, a.fp4, H, I, S, b4)) != MOE_OK) return st;
      if ((st = map_fp4_rows(&mA1, a.fp4 + off_w3, H, I, S, b4)) != MOE_OK) return st;
    } else {
      if ((st = map_fp4_rows(&mA0, a.fp4 + off_w2, I, H, S, b4)) != MOE_OK) return st;
      mA1 = mA0;
    }
  }
  if (sh) {
    if (mode == 0) {
      if ((st = map_u8_rows(&mS0, sh, H, I, 128)) != MOE_OK) return st;
      if ((st = map_u8_rows(&mS1, sh + f8_mat, H, I, 128)) != MOE_OK) return st;
    } else {
      if ((st = map_u8_rows(&mS0, sh + 2 * f8_mat, I, H, 128)) != MOE_OK) return st;
      mS1 = mS0;
    }
  }
  if (!a.fp4 || S == 0) {
    mA0 = mS0;
    mA1 = mS1;
  }
  if (!sh) {
    mS0 = mA0;
    mS1 = mA1;
  }
  if ((st = map_u8_rows(&mBh, mode == 0 ? b.xhi : b.hhi, a.K, rows, 16)) != MOE_OK) return st;
  if ((st = map_u8_rows(&mBl, mode == 0 ? b.xlo : b.hlo, a.K, rows, 16)) != MOE_OK) return st;

  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(mx8_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kM8Smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(mx8_gemm_kernel)");
    // all of the unified L1 / shared memory as shared memory, so two CTAs fit an SM
    e = cudaFuncSetAttribute(mx8_gemm_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(mx8_gemm_kernel carveout)");
    attr_set = true;
  }
  const long long items = (long long)max_groups * a.tiles;
  const int grid = (int)std::max(1LL, std::min<long long>((long long)kM8CtasPerSm * mx8_sm_count(), items));
  cudaError_t le = launch_pdl(mx8_gemm_kernel, dim3(grid), dim3(kM8Threads), (size_t)kM8Smem, stream, mA0, mA1, mS0,
                              mS1, mBh, mBl, a);
  if (le != cudaSuccess) return cuda_fail(le, mode == 0 ? "mx8_gemm_kernel (gate/up)" : "mx8_gemm_kernel (down)");
  return check_launch(mode == 0 ? "mx8_gemm_kernel (gate/up)" : "mx8_gemm_kernel (down)");
}

}  // namespace moe
