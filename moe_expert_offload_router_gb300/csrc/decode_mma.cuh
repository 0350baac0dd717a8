// Decode grouped expert MLP on the warp-level tensor-core MMA
// (mma.sync m16n8k16, f16 or bf16 operands, fp32 accumulate).
//
// "Running DeepSeek-V4-Flash across four free GPUs", section "What the expert
// cache actually does" (a grouped GEMM over the slot views, one expert's
// tokens together); "An elephant through a straw", sections "43 graphs, 43
// syncs" (grouped expert kernels per layer) and "Rig, model & methodology"
// (MXFP4 experts, one E8M0 scale per 32 weights, an FP8 shared expert).
//
// Decode batches give each expert a handful of tokens, so the layer streams
// its weights once and does little arithmetic per byte: the bound is HBM.  The
// weight tile is the MMA's A operand (M = weight rows), the group's tokens its
// B operand (N = 8 tokens), and A never touches shared memory: every thread
// loads 16 bytes of a weight row with one 128-bit load, converts its E2M1
// codes in registers (cvt.rn.f16x2.e2m1x2, then one fp16 multiply by the
// block scale) and feeds them straight to the MMA.  This works because a dot
// product may take its K terms in any order, as long as both operands use the
// same one.  In the fragment layout of m16n8k16, lane (g, q) = (lane / 4,
// lane % 4) holds the K slots {2q, 2q+1, 2q+8, 2q+9} of rows g and g+8; the K
// order used here gives MMA j of a 128-element chunk, in lane q, the elements
// 32q + 4j .. 32q + 4j + 3 of the chunk.  So a lane's 16 loaded bytes (one
// 32-weight block of one row: elements 32q .. 32q + 31) feed eight MMAs, and
// every K term of those MMAs in that lane shares the lane's block scale.  The
// activations are staged in shared memory in the same order (with a rotation
// of 16-byte units that keeps the 128-bit loads free of bank conflicts), so a
// lane reads the B fragments of two MMAs with one load.
//
// Work item: (token group of <= 16 tokens on one slot, tile of weight rows).
// A group's tokens are the N of up to two MMAs per A fragment, so a weight
// row is converted once for all of them.  Items are taken tile-major (all
// groups of tile 0, then of tile 1, ...), so the token groups of one popular
// expert read the same weight rows at about the same time and any repeated
// read hits L2.  A warp streams 4 weight rows (gate/up: rows f and f+8 of w1
// and of w3, so gate and up of a feature land in the same lane; down: rows f,
// f+8, f+16, f+24 of w2) one chunk at a time (128 elements of FP4, 64 of FP8:
// per lane 16 bytes of each row), with the next two chunks' loads in flight
// while one is computed.  The group's activations (16 tokens x K would fill
// the shared memory) pass through a double-buffered ring of 512-element K stages,
// filled with cp.async by all threads of the CTA one stage ahead; one barrier
// per stage.
//
// Precision: the E2M1 code times its E8M0 scale is exact in fp16 when the
// scale byte lies in [115, 140]; the activations are the fp16 copies scaled
// per token by a power of two (as in the CUDA-core kernels); products are
// exact and accumulate in fp32.  A chunk whose scales leave that
// range in any lane of the warp runs on bf16 operands instead (exact weights
// for every scale, activations converted back to bf16, which is exact for the
// bf16 inputs).  The FP8 shared expert's E4M3 codes are exact in fp16; its
// per-row scales multiply the fp32 accumulators.
//
// Included by expert_decode.cu (uses FwdArgs, Group, group_ok, ...).
#pragma once

namespace moe {

constexpr int kMmaWarps = 8;
constexpr int kMmaThreads = kMmaWarps * 32;
constexpr int kMmaFeat = 16 * kMmaWarps;       // gate/up features per item (of w1 and of w3)
constexpr int kMmaRowsDown = 32 * kMmaWarps;   // w2 rows per down item
constexpr int kMmaGroup = 16;                  // most tokens per group (two n8 tiles)
constexpr int kMmaStageK = 512;                // K elements per activation stage
// Stage row strides (bytes): FP4 layout (128-element chunks of four 32-element
// blocks) and FP8 layout (64-element chunks); the pads keep the 128-bit
// loads of a quarter warp on distinct banks.
constexpr int kMmaSrsFp4 = kMmaStageK * 2 + 32;
constexpr int kMmaSrsFp8 = kMmaStageK * 2 + 16;
constexpr int kMmaStageBytes = kMmaGroup * kMmaSrsFp4;
// shared memory: two stages, then tok[16], hrow[16] and the drawn item index
constexpr size_t kMmaSmem = 2 * (size_t)kMmaStageBytes + 3 * kMmaGroup * 4;

// Byte offset, within a staged row, of the 16-byte unit holding elements
// e .. e+7 (e a multiple of 8, counted from the stage's first element).
// FP4: chunk c = e / 128, block q, unit u; the unit sits at position
// (u + q / 2) mod 4 of its block.
__device__ __forceinline__ int mma_off_fp4(int e) {
  const int c = e >> 7, q = (e >> 5) & 3, u = (e >> 3) & 3;
  return c * 256 + q * 64 + (((u + (q >> 1)) & 3) << 4);
}
__device__ __forceinline__ int mma_off_fp8(int e) {
  const int c = e >> 6, q = (e >> 4) & 3, u = (e >> 3) & 1;
  return c * 128 + q * 32 + (u << 4);
}

__device__ __forceinline__ void mma_f16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(su32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// fp16 pair -> bf16 pair (exact for values with at most 8 significant bits)
__device__ __forceinline__ uint32_t h2_to_bf2(uint32_t h) {
  uint32_t r;
  asm("{\n\t.reg .b16 l, u, bl, bu;\n\tmov.b32 {l, u}, %1;\n\tcvt.rn.bf16.f16 bl, l;\n\tcvt.rn.bf16.f16 bu, u;\n\t"
      "mov.b32 %0, {bl, bu};\n\t}"
      : "=r"(r)
      : "r"(h));
  return r;
}
__device__ __forceinline__ uint32_t mul_h2(uint32_t a, uint32_t s) {
  __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&s));
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t mul_bf2(uint32_t a, uint32_t s) {
  __nv_bfloat162 v =
      __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&a), *reinterpret_cast<const __nv_bfloat162*>(&s));
  return *reinterpret_cast<uint32_t*>(&v);
}

// E8M0 scale byte as an fp16 pair (a normal fp16 for bytes 113 .. 142) and as a
// bf16 pair (every byte; 0 is the subnormal 2^-127).
constexpr uint32_t kMmaF16Lo = 115, kMmaF16Hi = 140;
__device__ __forceinline__ uint32_t scale_h2(uint32_t e) {
  const uint32_t h = (e - 112u) << 10;
  return h | (h << 16);
}
__device__ __forceinline__ uint32_t scale_bf2(uint32_t e) {
  const uint32_t b = e ? (e << 7) : 0x0040u;
  return b | (b << 16);
}
__device__ __forceinline__ bool byte_in(uint32_t w, int sh) {
  const uint32_t e = (w >> sh) & 0xffu;
  return e >= kMmaF16Lo && e <= kMmaF16Hi;
}

// Rows of one warp: row r's codes at cb + co[r], its scales at sb + so[r]
// (byte offsets within one expert, so 32 bits hold them).
struct MmaRows {
  const uint8_t* cb;
  const uint8_t* sb;
  uint32_t co[4], so[4];
};

// One chunk of four weight rows: this lane's 16 code bytes of each row, and
// (FP4) the row's four scale bytes of the chunk (blocks 4c .. 4c+3; the lane
// uses byte q).
struct MmaChunk {
  uint4 q[4];
  uint32_t s[4];
};

template <bool FP8>
__device__ __forceinline__ void mma_load(MmaChunk& b, const MmaRows& w, int c, int q) {
  const uint8_t* cp = w.cb + (size_t)c * 64 + 16 * q;
#pragma unroll
  for (int r = 0; r < 4; ++r) b.q[r] = ld_stream_v4(cp + w.co[r]);
  if (!FP8) {
    const uint8_t* sp = w.sb + 4 * c;
#pragma unroll
    for (int r = 0; r < 4; ++r) b.s[r] = __ldg(reinterpret_cast<const uint32_t*>(sp + w.so[r]));
  }
}

// Adds one FP4 chunk's products for NB n8 token tiles: rows 0 and 1 (weight rows
// f, f+8) into a0[t], rows 2 and 3 into a1[t].  brow: the staged row of token g
// of tile 0 (tile t at + 8 t rows); lc: the chunk's index within the stage.
template <int NB, bool F16>
__device__ __forceinline__ void mma_fp4_compute(const MmaChunk& b, const uint8_t* brow, int lc, int q, int nt,
                                                float (&a0)[NB][4], float (&a1)[NB][4]) {
  uint32_t sc[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const uint32_t e = (b.s[r] >> (8 * q)) & 0xffu;
    sc[r] = F16 ? scale_h2(e) : scale_bf2(e);
  }
  const uint8_t* bp = brow + lc * 256 + q * 64;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t h[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const uint32_t word = w == 0 ? b.q[r].x : w == 1 ? b.q[r].y : w == 2 ? b.q[r].z : b.q[r].w;
      __half2 t[4];
      fp4_word_to_h2(word, t);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t v = *reinterpret_cast<uint32_t*>(&t[u]);
        h[r][u] = F16 ? mul_h2(v, sc[r]) : mul_bf2(h2_to_bf2(v), sc[r]);
      }
    }
    // code word w holds the lane's elements 8w .. 8w+7 of its block: MMA 2w
    // takes bytes 0 and 1 (a0/a2 of rows f and f+8), MMA 2w+1 bytes 2 and 3
#pragma unroll
    for (int t = 0; t < NB; ++t) {
      if (t >= nt) break;  // tiles past the group's tokens (warp-uniform)
      uint4 bv = lds128(bp + t * 8 * kMmaSrsFp4 + (((w + (q >> 1)) & 3) << 4));
      if (F16) {
        mma_f16(a0[t], h[0][0], h[1][0], h[0][1], h[1][1], bv.x, bv.y);
        mma_f16(a1[t], h[2][0], h[3][0], h[2][1], h[3][1], bv.x, bv.y);
        mma_f16(a0[t], h[0][2], h[1][2], h[0][3], h[1][3], bv.z, bv.w);
        mma_f16(a1[t], h[2][2], h[3][2], h[2][3], h[3][3], bv.z, bv.w);
      } else {
        bv.x = h2_to_bf2(bv.x);
        bv.y = h2_to_bf2(bv.y);
        bv.z = h2_to_bf2(bv.z);
        bv.w = h2_to_bf2(bv.w);
        mma_bf16(a0[t], h[0][0], h[1][0], h[0][1], h[1][1], bv.x, bv.y);
        mma_bf16(a1[t], h[2][0], h[3][0], h[2][1], h[3][1], bv.x, bv.y);
        mma_bf16(a0[t], h[0][2], h[1][2], h[0][3], h[1][3], bv.z, bv.w);
        mma_bf16(a1[t], h[2][2], h[3][2], h[2][3], h[3][3], bv.z, bv.w);
      }
    }
  }
}

// FP8 (E4M3, the shared expert): code word w of a row holds the lane's elements
// 4w .. 4w+3 of its 16-element block, the operands of MMA w of the chunk.
template <int NB>
__device__ __forceinline__ void mma_fp8_compute(const MmaChunk& b, const uint8_t* brow, int lc, int q, int nt,
                                                float (&a0)[NB][4], float (&a1)[NB][4]) {
  const uint8_t* bp = brow + lc * 128 + q * 32;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
#pragma unroll
    for (int hw = 0; hw < 2; ++hw) {
      const int w = 2 * u + hw;
      uint32_t a[4][2];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t word = w == 0 ? b.q[r].x : w == 1 ? b.q[r].y : w == 2 ? b.q[r].z : b.q[r].w;
        const __half2 lo = e4m3x2_to_h2(word & 0xffffu), hi = e4m3x2_to_h2(word >> 16);
        a[r][0] = *reinterpret_cast<const uint32_t*>(&lo);
        a[r][1] = *reinterpret_cast<const uint32_t*>(&hi);
      }
#pragma unroll
      for (int t = 0; t < NB; ++t) {
        if (t >= nt) break;
        const uint4 bv = lds128(bp + t * 8 * kMmaSrsFp8 + 16 * u);
        const uint32_t b0 = hw ? bv.z : bv.x, b1 = hw ? bv.w : bv.y;
        mma_f16(a0[t], a[0][0], a[1][0], a[0][1], a[1][1], b0, b1);
        mma_f16(a1[t], a[2][0], a[3][0], a[2][1], a[3][1], b0, b1);
      }
    }
  }
}

// The whole K of four weight rows against the group's activations, streamed
// through the two-stage ring (stage s in buffer s % 2; stage 0 already issued
// by the caller; issue(s) fills stage s).  A ring of R chunk buffers keeps the
// next R - 1 chunks' weight loads in flight while a chunk is computed: three
// for one token tile, two for more (a chunk's compute is then longer, and the
// accumulators need the registers).  The barrier at each stage's first chunk
// makes that stage visible to every warp and frees the other buffer (every warp
// has finished the previous stage) for the next stage's copies.  K is a
// multiple of kMmaStageK.
template <int NB, bool FP8, class Issue>
__device__ __forceinline__ void mma_rows(const MmaRows& rw, int K, const uint8_t* stages, int g, int q, int nt,
                                         float (&a0)[NB][4], float (&a1)[NB][4], Issue issue) {
  constexpr int R = NB == 1 ? 3 : 2;          // chunk buffers
  constexpr int CK = FP8 ? 64 : 128;          // K elements per chunk
  constexpr int CPS = kMmaStageK / CK;        // chunks per stage
  constexpr int SRS = FP8 ? kMmaSrsFp8 : kMmaSrsFp4;
  const int nch = K / CK, nst = K / kMmaStageK;
  MmaChunk b[R];
#pragma unroll
  for (int j = 0; j + 1 < R; ++j) mma_load<FP8>(b[j], rw, j, q);
  for (int c0 = 0; c0 < nch; c0 += R) {
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int c = c0 + j;
      if (c >= nch) break;
      if (c + R - 1 < nch) mma_load<FP8>(b[(j + R - 1) % R], rw, c + R - 1, q);
      const int s = c / CPS, lc = c - s * CPS;
      if (lc == 0) {
        cp_async_wait_all();
        __syncthreads();
        if (s + 1 < nst) issue(s + 1);
      }
      const uint8_t* brow = stages + (size_t)(s & 1) * kMmaStageBytes + g * SRS;
      if (FP8) {
        mma_fp8_compute<NB>(b[j], brow, lc, q, nt, a0, a1);
      } else {
        bool ok = true;
#pragma unroll
        for (int r = 0; r < 4; ++r) ok = ok && byte_in(b[j].s[r], 8 * q);
        if (__all_sync(0xffffffffu, ok))
          mma_fp4_compute<NB, true>(b[j], brow, lc, q, nt, a0, a1);
        else
          mma_fp4_compute<NB, false>(b[j], brow, lc, q, nt, a0, a1);
      }
    }
  }
}

// Copies stage s (elements [s * kMmaStageK, (s + 1) * kMmaStageK)) of the n
// fp16 rows src + row[i] * ld into buf, in the format's layout; one commit group.
__device__ __forceinline__ void mma_issue_stage(uint8_t* buf, const __half* src, const int* row, int ld, int n,
                                                int s, bool fp8) {
  constexpr int units = kMmaStageK / 8;
  const int srs = fp8 ? kMmaSrsFp8 : kMmaSrsFp4;
  for (int v = threadIdx.x; v < n * units; v += kMmaThreads) {
    const int i = v / units, e = (v - i * units) * 8;
    cp_async16(buf + i * srs + (fp8 ? mma_off_fp8(e) : mma_off_fp4(e)),
               src + (size_t)row[i] * ld + (size_t)s * kMmaStageK + e);
  }
  cp_async_commit();
}

// Pools the warp-MMA kernels take (bit per pool); the CUDA-core kernels skip them.
constexpr int kMmaPoolMask = (1 << MOE_POOL_FP4) | (1 << MOE_POOL_SHARED);

template <int NB>
__device__ __forceinline__ void zero_acc(float (&a)[NB][4]) {
#pragma unroll
  for (int t = 0; t < NB; ++t) a[t][0] = a[t][1] = a[t][2] = a[t][3] = 0.f;
}

// ------------------------------------------------------------ gate/up + SwiGLU --
template <int NB>
__device__ __forceinline__ void mma_gateup_item(const FwdArgs& a, const Group& grp, const MatView& w1,
                                                const MatView& w3, int f, uint8_t* smem, const int* tok,
                                                const int* hrow) {
  const int H = a.H, I = a.I;
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const bool fp8 = grp.pool == MOE_POOL_SHARED;
  const uint32_t rb = fp8 ? H : H / 2;  // code bytes per row
  MmaRows rw;
  rw.cb = w1.codes;
  rw.sb = w1.scales;
  const uint32_t m3c = (uint32_t)(w3.codes - w1.codes), m3s = (uint32_t)(w3.scales - w1.scales);
  rw.co[0] = f * rb;
  rw.co[1] = (f + 8) * rb;
  rw.co[2] = m3c + f * rb;
  rw.co[3] = m3c + (f + 8) * rb;
  rw.so[0] = f * (H / 32);
  rw.so[1] = (f + 8) * (H / 32);
  rw.so[2] = m3s + f * (H / 32);
  rw.so[3] = m3s + (f + 8) * (H / 32);
  float ag[NB][4], au[NB][4];
  zero_acc<NB>(ag);
  zero_acc<NB>(au);
  auto issue = [&](int s) { mma_issue_stage(smem + (s & 1) * kMmaStageBytes, a.xs, tok, H, grp.count, s, fp8); };
  issue(0);
  const int nt = (grp.count + 7) / 8;
  if (fp8)
    mma_rows<NB, true>(rw, H, smem, g, q, nt, ag, au, issue);
  else
    mma_rows<NB, false>(rw, H, smem, g, q, nt, ag, au, issue);
  // lane holds (row f + 8 hr, token 8 t + 2 q + tt) at [t][2 hr + tt]
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int feat = f + 8 * hr;
    const float rg = fp8 ? __ldg(reinterpret_cast<const float*>(w1.scales) + feat) : 1.f;
    const float ru = fp8 ? __ldg(reinterpret_cast<const float*>(w3.scales) + feat) : 1.f;
#pragma unroll
    for (int t = 0; t < NB; ++t)
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        const int i = 8 * t + 2 * q + tt;
        if (i < grp.count) {
          const int sg = a.xsig[tok[i]];
          const float gv = ldexpf(ag[t][2 * hr + tt] * rg, sg);
          const float uv = ldexpf(au[t][2 * hr + tt] * ru, sg);
          a.h[(size_t)hrow[i] * I + feat] = gv / (1.f + expf(-gv)) * uv;
        }
      }
  }
}

// Items are handed out by a counter (a.hdr[2], zeroed by the plan kernel), so
// a CTA that drew cheap items takes more; item i is tile i / ngroups and group
// ngroups - 1 - i % ngroups (the shared expert's groups, last in the list and
// twice the bytes per row, come first in each tile).
__device__ __forceinline__ long long mma_next_item(int* counter, int* slot) {
  __syncthreads();  // the previous item is done with the stages and the row lists
  if (threadIdx.x == 0) *slot = atomicAdd(counter, 1);
  __syncthreads();
  return *slot;
}

// NB: token tiles of a group (groups of up to 8 NB tokens), one per launch.
template <int NB>
__global__ void __launch_bounds__(kMmaThreads, 2) mma_gateup_kernel(FwdArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int H = a.H, I = a.I;
  int* tok = reinterpret_cast<int*>(smem_raw + 2 * (size_t)kMmaStageBytes);
  int* hrow = tok + kMmaGroup;
  int* slot = hrow + kMmaGroup;
  const int warp = threadIdx.x >> 5, g = (threadIdx.x & 31) >> 2;
  const int tiles = I / kMmaFeat;
  const int ngr = n_groups_checked(a);
  const long long n_items = (long long)ngr * tiles;
  for (;;) {
    const long long item = mma_next_item(a.hdr + 2, slot);
    if (item >= n_items) break;
    const int tile = (int)(item / ngr), gi = ngr - 1 - (int)(item % ngr);
    const Group grp = a.groups[gi];
    if (grp.pool < 0 || grp.pool > 2 || !((kMmaPoolMask >> grp.pool) & 1)) continue;  // 2-bit: the CUDA-core kernel's
    if (!group_ok(a, grp)) {
      if (threadIdx.x == 0 && a.err) *a.err = MOE_ERR_INVALID;
      continue;
    }
    const bool fp8 = grp.pool == MOE_POOL_SHARED;
    const uint8_t* ex = expert_base(a, grp.pool, grp.slot);
    const MatView w1 = mat_view(grp.pool, ex, H, I, 0), w3 = mat_view(grp.pool, ex, H, I, 1);
    const int f = tile * kMmaFeat + warp * 16 + g;  // this lane's rows: f and f + 8
    if (threadIdx.x < grp.count) {
      const int i = threadIdx.x;
      if (fp8) {
        tok[i] = grp.begin + i;
        hrow[i] = a.P + grp.begin + i;
      } else {
        const int p = min(max(a.perm[grp.begin + i], 0), a.P - 1);
        tok[i] = p / a.k;
        hrow[i] = p;
      }
    }
    __syncthreads();
    mma_gateup_item<NB>(a, grp, w1, w3, f, smem_raw, tok, hrow);
  }
}

// ------------------------------------------------------------------- h prep --
// One warp per row of h (fp32 [rows, I]): the power-of-two exponent that brings
// the row's largest magnitude into [1, 2), and the row in fp16 times 2^-exponent
// (the down kernels' activations).
__global__ void __launch_bounds__(256) mma_hprep_kernel(const float* h, int rows, int I, __half* hs, int* hsig) {
  const int lane = threadIdx.x & 31;
  for (int r = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5); r < rows;
       r += (int)((gridDim.x * (size_t)blockDim.x) >> 5)) {
    const float* src = h + (size_t)r * I;
    float m = 0.f;
    for (int n = 4 * lane; n < I; n += 128) {
      const float4 v = *reinterpret_cast<const float4*>(src + n);
      m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int sg = pow2_exponent(m);
    if (lane == 0) hsig[r] = sg;
    __half* dst = hs + (size_t)r * I;
    for (int n = 8 * lane; n < I; n += 256) {
      const float4 v0 = *reinterpret_cast<const float4*>(src + n);
      const float4 v1 = *reinterpret_cast<const float4*>(src + n + 4);
      __half2 hv[4];
      hv[0] = __floats2half2_rn(ldexpf(v0.x, -sg), ldexpf(v0.y, -sg));
      hv[1] = __floats2half2_rn(ldexpf(v0.z, -sg), ldexpf(v0.w, -sg));
      hv[2] = __floats2half2_rn(ldexpf(v1.x, -sg), ldexpf(v1.y, -sg));
      hv[3] = __floats2half2_rn(ldexpf(v1.z, -sg), ldexpf(v1.w, -sg));
      *reinterpret_cast<uint4*>(dst + n) = *reinterpret_cast<uint4*>(hv);
    }
  }
}

// ---------------------------------------------------------------------- down --
template <int NB>
__device__ __forceinline__ void mma_down_item(const FwdArgs& a, const Group& grp, const MatView& w2, int f,
                                              uint8_t* smem, const int* hrow) {
  const int H = a.H, I = a.I;
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const bool fp8 = grp.pool == MOE_POOL_SHARED;
  const uint32_t rb = fp8 ? I : I / 2;
  MmaRows rw;
  rw.cb = w2.codes;
  rw.sb = w2.scales;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    rw.co[r] = (f + 8 * r) * rb;
    rw.so[r] = (f + 8 * r) * (I / 32);
  }
  float a0[NB][4], a1[NB][4];
  zero_acc<NB>(a0);
  zero_acc<NB>(a1);
  auto issue = [&](int s) { mma_issue_stage(smem + (s & 1) * kMmaStageBytes, a.hs16, hrow, I, grp.count, s, fp8); };
  issue(0);
  const int nt = (grp.count + 7) / 8;
  if (fp8)
    mma_rows<NB, true>(rw, I, smem, g, q, nt, a0, a1, issue);
  else
    mma_rows<NB, false>(rw, I, smem, g, q, nt, a0, a1, issue);
#pragma unroll
  for (int hr = 0; hr < 4; ++hr) {
    const int row = f + 8 * hr;
    const float rw2 = fp8 ? __ldg(reinterpret_cast<const float*>(w2.scales) + row) : 1.f;
#pragma unroll
    for (int t = 0; t < NB; ++t)
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        const int i = 8 * t + 2 * q + tt;
        if (i < grp.count) {
          const float v = (hr < 2 ? a0[t][2 * hr + tt] : a1[t][2 * (hr - 2) + tt]);
          a.o[(size_t)hrow[i] * H + row] = ldexpf(v * rw2, a.hsig[hrow[i]]);
        }
      }
  }
}

template <int NB>
__global__ void __launch_bounds__(kMmaThreads, 2) mma_down_kernel(FwdArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int H = a.H, I = a.I;
  int* hrow = reinterpret_cast<int*>(smem_raw + 2 * (size_t)kMmaStageBytes);
  int* slot = hrow + 2 * kMmaGroup;
  const int warp = threadIdx.x >> 5, g = (threadIdx.x & 31) >> 2;
  const int tiles = H / kMmaRowsDown;
  const int ngr = n_groups_checked(a);
  const long long n_items = (long long)ngr * tiles;
  for (;;) {
    const long long item = mma_next_item(a.hdr + 3, slot);
    if (item >= n_items) break;
    const int tile = (int)(item / ngr), gi = ngr - 1 - (int)(item % ngr);
    const Group grp = a.groups[gi];
    if (grp.pool < 0 || grp.pool > 2 || !((kMmaPoolMask >> grp.pool) & 1)) continue;
    if (!group_ok(a, grp)) {
      if (threadIdx.x == 0 && a.err) *a.err = MOE_ERR_INVALID;
      continue;
    }
    const uint8_t* ex = expert_base(a, grp.pool, grp.slot);
    const MatView w2 = mat_view(grp.pool, ex, H, I, 2);
    const int f = tile * kMmaRowsDown + warp * 32 + g;  // rows f, f+8, f+16, f+24
    if (threadIdx.x < grp.count) {
      const int i = threadIdx.x;
      hrow[i] = grp.pool == MOE_POOL_SHARED ? a.P + grp.begin + i : min(max(a.perm[grp.begin + i], 0), a.P - 1);
    }
    __syncthreads();
    mma_down_item<NB>(a, grp, w2, f, smem_raw, hrow);
  }
}

}  // namespace moe
