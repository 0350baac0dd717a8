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
// activations are staged once per item in shared memory in the same order
// (with a rotation of 16-byte units that keeps the 128-bit loads free of bank
// conflicts), so a lane reads the B fragments of two MMAs with one load.
//
// Work item: (token group of <= 8 tokens on one slot, tile of weight rows).
// Items are taken tile-major (all groups of tile 0, then of tile 1, ...), so the
// token groups of one popular expert read the same weight rows at about the
// same time and the repeated reads hit L2.  A warp streams 4 weight rows
// (gate/up: rows f and f+8 of w1 and of w3, so gate and up of a feature land in
// the same lane; down: rows f, f+8, f+16, f+24 of w2) two 128-element chunks
// at a time (a 128-element chunk of FP4, 64 of FP8, per lane 16 bytes of each
// row), with the next two chunks' loads in flight while one is computed.
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

// Staged activation row stride (bytes) for K elements: FP4 layout (128-element
// chunks of four 32-element blocks) and FP8 layout (64-element chunks).
__host__ __device__ constexpr int mma_rs_fp4(int K) { return K * 2 + 32; }
__host__ __device__ constexpr int mma_rs_fp8(int K) { return K * 2 + 16; }

// Byte offset, within a staged row, of the 16-byte unit holding elements
// e .. e+7 (e a multiple of 8).  FP4: chunk c = e / 128, block q, unit u;
// the unit sits at position (u + q / 2) mod 4 of its block.
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

// One 128-element chunk of four weight rows (FP4): this lane's 16 code bytes of
// each row and the row's four scale bytes of the chunk (blocks 4c .. 4c+3; the
// lane uses byte q).
struct MmaFp4Chunk {
  uint4 q[4];
  uint32_t s[4];
};

// Rows of one warp: row r's codes at cb + co[r], its scales at sb + so[r]
// (byte offsets within one expert, so 32 bits hold them).
struct MmaRows {
  const uint8_t* cb;
  const uint8_t* sb;
  uint32_t co[4], so[4];
};

__device__ __forceinline__ void mma_fp4_load(MmaFp4Chunk& b, const MmaRows& w, int c, int q) {
  const uint8_t* cp = w.cb + (size_t)c * 64 + 16 * q;
  const uint8_t* sp = w.sb + 4 * c;
#pragma unroll
  for (int r = 0; r < 4; ++r) b.q[r] = ld_stream_v4(cp + w.co[r]);
#pragma unroll
  for (int r = 0; r < 4; ++r) b.s[r] = __ldg(reinterpret_cast<const uint32_t*>(sp + w.so[r]));
}

// Adds one chunk's products: rows 0 and 1 (weight rows f, f+8) into acc0, rows
// 2 and 3 into acc1.  brow: the staged activation row of token g.
template <bool F16>
__device__ __forceinline__ void mma_fp4_compute(const MmaFp4Chunk& b, const uint8_t* brow, int c, int q, float* acc0,
                                                float* acc1) {
  uint32_t sc[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const uint32_t e = (b.s[r] >> (8 * q)) & 0xffu;
    sc[r] = F16 ? scale_h2(e) : scale_bf2(e);
  }
  const uint8_t* bp = brow + c * 256 + q * 64;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint4 bv = lds128(bp + (((w + (q >> 1)) & 3) << 4));
    if (!F16) {
      bv.x = h2_to_bf2(bv.x);
      bv.y = h2_to_bf2(bv.y);
      bv.z = h2_to_bf2(bv.z);
      bv.w = h2_to_bf2(bv.w);
    }
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
    if (F16) {
      mma_f16(acc0, h[0][0], h[1][0], h[0][1], h[1][1], bv.x, bv.y);
      mma_f16(acc1, h[2][0], h[3][0], h[2][1], h[3][1], bv.x, bv.y);
      mma_f16(acc0, h[0][2], h[1][2], h[0][3], h[1][3], bv.z, bv.w);
      mma_f16(acc1, h[2][2], h[3][2], h[2][3], h[3][3], bv.z, bv.w);
    } else {
      mma_bf16(acc0, h[0][0], h[1][0], h[0][1], h[1][1], bv.x, bv.y);
      mma_bf16(acc1, h[2][0], h[3][0], h[2][1], h[3][1], bv.x, bv.y);
      mma_bf16(acc0, h[0][2], h[1][2], h[0][3], h[1][3], bv.z, bv.w);
      mma_bf16(acc1, h[2][2], h[3][2], h[2][3], h[3][3], bv.z, bv.w);
    }
  }
}

// fp16 operands when every lane's block scales of the chunk allow them
__device__ __forceinline__ void mma_fp4_chunk(const MmaFp4Chunk& b, const uint8_t* brow, int c, int q, float* acc0,
                                              float* acc1) {
  bool ok = true;
#pragma unroll
  for (int r = 0; r < 4; ++r) ok = ok && byte_in(b.s[r], 8 * q);
  if (__all_sync(0xffffffffu, ok))
    mma_fp4_compute<true>(b, brow, c, q, acc0, acc1);
  else
    mma_fp4_compute<false>(b, brow, c, q, acc0, acc1);
}

// Four FP4 weight rows (codes crow[r], scales srow[r], K elements each) against
// the staged activations of the group: acc0 += rows 0/1, acc1 += rows 2/3.  K
// is a multiple of 128.  A ring of three chunk buffers keeps the next two
// chunks' loads in flight while a chunk is computed.
__device__ __forceinline__ void mma_fp4_rows(const MmaRows& rw, int K, const uint8_t* brow, float* acc0,
                                             float* acc1) {
  const int q = threadIdx.x & 3;
  const int nch = K / 128;
  MmaFp4Chunk b0, b1, b2;
  mma_fp4_load(b0, rw, 0, q);
  if (nch > 1) mma_fp4_load(b1, rw, 1, q);
  for (int c = 0; c < nch; c += 3) {
    if (c + 2 < nch) mma_fp4_load(b2, rw, c + 2, q);
    mma_fp4_chunk(b0, brow, c, q, acc0, acc1);
    if (c + 1 >= nch) break;
    if (c + 3 < nch) mma_fp4_load(b0, rw, c + 3, q);
    mma_fp4_chunk(b1, brow, c + 1, q, acc0, acc1);
    if (c + 2 >= nch) break;
    if (c + 4 < nch) mma_fp4_load(b1, rw, c + 4, q);
    mma_fp4_chunk(b2, brow, c + 2, q, acc0, acc1);
  }
}

// FP8 (E4M3, the shared expert): 64-element chunks, 16 codes per lane per row.
struct MmaFp8Chunk {
  uint4 q[4];
};

__device__ __forceinline__ void mma_fp8_load(MmaFp8Chunk& b, const MmaRows& w, int c, int q) {
  const uint8_t* cp = w.cb + (size_t)c * 64 + 16 * q;
#pragma unroll
  for (int r = 0; r < 4; ++r) b.q[r] = ld_stream_v4(cp + w.co[r]);
}

__device__ __forceinline__ void mma_fp8_compute(const MmaFp8Chunk& b, const uint8_t* brow, int c, int q, float* acc0,
                                                float* acc1) {
  const uint8_t* bp = brow + c * 128 + q * 32;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const uint4 bv = lds128(bp + 16 * u);
#pragma unroll
    for (int hw = 0; hw < 2; ++hw) {  // MMA 2u + hw: code word 2u + hw of each row (elements 4w .. 4w+3)
      const int w = 2 * u + hw;
      uint32_t a[4][2];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t word = w == 0 ? b.q[r].x : w == 1 ? b.q[r].y : w == 2 ? b.q[r].z : b.q[r].w;
        const __half2 lo = e4m3x2_to_h2(word & 0xffffu), hi = e4m3x2_to_h2(word >> 16);
        a[r][0] = *reinterpret_cast<const uint32_t*>(&lo);
        a[r][1] = *reinterpret_cast<const uint32_t*>(&hi);
      }
      const uint32_t b0 = hw ? bv.z : bv.x, b1 = hw ? bv.w : bv.y;
      mma_f16(acc0, a[0][0], a[1][0], a[0][1], a[1][1], b0, b1);
      mma_f16(acc1, a[2][0], a[3][0], a[2][1], a[3][1], b0, b1);
    }
  }
}

// K a multiple of 64.
__device__ __forceinline__ void mma_fp8_rows(const MmaRows& rw, int K, const uint8_t* brow, float* acc0,
                                             float* acc1) {
  const int q = threadIdx.x & 3;
  const int nch = K / 64;
  MmaFp8Chunk b0, b1, b2;
  mma_fp8_load(b0, rw, 0, q);
  if (nch > 1) mma_fp8_load(b1, rw, 1, q);
  for (int c = 0; c < nch; c += 3) {
    if (c + 2 < nch) mma_fp8_load(b2, rw, c + 2, q);
    mma_fp8_compute(b0, brow, c, q, acc0, acc1);
    if (c + 1 >= nch) break;
    if (c + 3 < nch) mma_fp8_load(b0, rw, c + 3, q);
    mma_fp8_compute(b1, brow, c + 1, q, acc0, acc1);
    if (c + 2 >= nch) break;
    if (c + 4 < nch) mma_fp8_load(b1, rw, c + 4, q);
    mma_fp8_compute(b2, brow, c + 2, q, acc0, acc1);
  }
}

// Pools the warp-MMA kernels take (bit per pool); the CUDA-core kernels skip them.
constexpr int kMmaPoolMask = (1 << MOE_POOL_FP4) | (1 << MOE_POOL_SHARED);

__device__ __forceinline__ long long mma_item_count(const FwdArgs& a, int tiles, int* n_groups) {
  *n_groups = n_groups_checked(a);
  return (long long)(*n_groups) * tiles;
}

// ------------------------------------------------------------ gate/up + SwiGLU --
// Smem: kG staged rows (each format at its own stride; the FP4 one is the
// larger), then tok[kG], hrow[kG].
__global__ void __launch_bounds__(kMmaThreads, 2) mma_gateup_kernel(FwdArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int H = a.H, I = a.I;
  const int RS = mma_rs_fp4(H);
  int* tok = reinterpret_cast<int*>(smem_raw + (size_t)kG * RS);
  int* hrow = tok + kG;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int tiles = I / kMmaFeat;
  int ngr;
  const long long n_items = mma_item_count(a, tiles, &ngr);
  for (long long item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int tile = (int)(item / ngr), gi = (int)(item % ngr);
    const Group grp = a.groups[gi];
    if (!((kMmaPoolMask >> grp.pool) & 1)) continue;  // a 2-bit group: the CUDA-core kernel's
    if (!group_ok(a, grp)) {
      if (threadIdx.x == 0 && a.err) *a.err = MOE_ERR_INVALID;
      continue;
    }
    const bool fp8 = grp.pool == MOE_POOL_SHARED;
    const int rs = fp8 ? mma_rs_fp8(H) : RS;
    const uint8_t* ex = expert_base(a, grp.pool, grp.slot);
    const MatView w1 = mat_view(grp.pool, ex, H, I, 0), w3 = mat_view(grp.pool, ex, H, I, 1);
    const int f = tile * kMmaFeat + warp * 16 + g;  // this lane's rows: f and f + 8
    const uint32_t rb = fp8 ? H : H / 2;            // code bytes per row
    MmaRows rw;
    rw.cb = w1.codes;
    rw.sb = w1.scales;
    {
      const uint32_t m3c = (uint32_t)(w3.codes - w1.codes), m3s = (uint32_t)(w3.scales - w1.scales);
      rw.co[0] = f * rb;
      rw.co[1] = (f + 8) * rb;
      rw.co[2] = m3c + f * rb;
      rw.co[3] = m3c + (f + 8) * rb;
      rw.so[0] = f * (H / 32);
      rw.so[1] = (f + 8) * (H / 32);
      rw.so[2] = m3s + f * (H / 32);
      rw.so[3] = m3s + (f + 8) * (H / 32);
    }
    __syncthreads();  // the previous item is done with the staged rows
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
    {
      const int units = H / 8;
      for (int v = threadIdx.x; v < grp.count * units; v += blockDim.x) {
        const int i = v / units, e = (v - i * units) * 8;
        const uint4 val = *reinterpret_cast<const uint4*>(a.xs + (size_t)tok[i] * H + e);
        *reinterpret_cast<uint4*>(smem_raw + (size_t)i * rs + (fp8 ? mma_off_fp8(e) : mma_off_fp4(e))) = val;
      }
    }
    __syncthreads();
    float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
    const uint8_t* brow = smem_raw + (size_t)g * rs;
    if (fp8)
      mma_fp8_rows(rw, H, brow, ag, au);
    else
      mma_fp4_rows(rw, H, brow, ag, au);
    // lane holds (row f + 8 hr, token 2q + t) at index 2 hr + t
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int feat = f + 8 * hr;
      const float rg = fp8 ? __ldg(reinterpret_cast<const float*>(w1.scales) + feat) : 1.f;
      const float ru = fp8 ? __ldg(reinterpret_cast<const float*>(w3.scales) + feat) : 1.f;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int i = 2 * q + t;
        if (i < grp.count) {
          const int sg = a.xsig[tok[i]];
          const float gv = ldexpf(ag[2 * hr + t] * rg, sg);
          const float uv = ldexpf(au[2 * hr + t] * ru, sg);
          a.h[(size_t)hrow[i] * I + feat] = gv / (1.f + expf(-gv)) * uv;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------- down --
// Smem: kG staged rows of h (fp16, per-pair power-of-two scale), hrow[kG], sig[kG].
__global__ void __launch_bounds__(kMmaThreads, 2) mma_down_kernel(FwdArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int H = a.H, I = a.I;
  const int RS = mma_rs_fp4(I);
  int* hrow = reinterpret_cast<int*>(smem_raw + (size_t)kG * RS);
  int* sig = hrow + kG;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int tiles = H / kMmaRowsDown;
  int ngr;
  const long long n_items = mma_item_count(a, tiles, &ngr);
  for (long long item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int tile = (int)(item / ngr), gi = (int)(item % ngr);
    const Group grp = a.groups[gi];
    if (!((kMmaPoolMask >> grp.pool) & 1)) continue;
    if (!group_ok(a, grp)) {
      if (threadIdx.x == 0 && a.err) *a.err = MOE_ERR_INVALID;
      continue;
    }
    const bool fp8 = grp.pool == MOE_POOL_SHARED;
    const int rs = fp8 ? mma_rs_fp8(I) : RS;
    const uint8_t* ex = expert_base(a, grp.pool, grp.slot);
    const MatView w2 = mat_view(grp.pool, ex, H, I, 2);
    const int f = tile * kMmaRowsDown + warp * 32 + g;  // rows f, f+8, f+16, f+24
    const uint32_t rb = fp8 ? I : I / 2;
    MmaRows rw;
    rw.cb = w2.codes;
    rw.sb = w2.scales;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      rw.co[r] = (f + 8 * r) * rb;
      rw.so[r] = (f + 8 * r) * (I / 32);
    }
    __syncthreads();
    if (threadIdx.x < grp.count) {
      const int i = threadIdx.x;
      hrow[i] = fp8 ? a.P + grp.begin + i : min(max(a.perm[grp.begin + i], 0), a.P - 1);
    }
    __syncthreads();
    // one warp per row of h: power-of-two scale of its largest magnitude, then fp16
    for (int i = warp; i < grp.count; i += kMmaWarps) {
      const float* src = a.h + (size_t)hrow[i] * I;
      float m = 0.f;
      for (int n = 4 * lane; n < I; n += 128) {
        const float4 v = *reinterpret_cast<const float4*>(src + n);
        m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      const int sg = pow2_exponent(m);
      if (lane == 0) sig[i] = sg;
      uint8_t* dst = smem_raw + (size_t)i * rs;
      for (int e = 8 * lane; e < I; e += 256) {
        const float4 v0 = *reinterpret_cast<const float4*>(src + e);
        const float4 v1 = *reinterpret_cast<const float4*>(src + e + 4);
        __half2 hv[4];
        hv[0] = __floats2half2_rn(ldexpf(v0.x, -sg), ldexpf(v0.y, -sg));
        hv[1] = __floats2half2_rn(ldexpf(v0.z, -sg), ldexpf(v0.w, -sg));
        hv[2] = __floats2half2_rn(ldexpf(v1.x, -sg), ldexpf(v1.y, -sg));
        hv[3] = __floats2half2_rn(ldexpf(v1.z, -sg), ldexpf(v1.w, -sg));
        *reinterpret_cast<uint4*>(dst + (fp8 ? mma_off_fp8(e) : mma_off_fp4(e))) = *reinterpret_cast<uint4*>(hv);
      }
    }
    __syncthreads();
    float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
    const uint8_t* brow = smem_raw + (size_t)g * rs;
    if (fp8)
      mma_fp8_rows(rw, I, brow, a0, a1);
    else
      mma_fp4_rows(rw, I, brow, a0, a1);
#pragma unroll
    for (int hr = 0; hr < 4; ++hr) {
      const int row = f + 8 * hr;
      const float rw = fp8 ? __ldg(reinterpret_cast<const float*>(w2.scales) + row) : 1.f;
      const float* acc = hr < 2 ? a0 : a1;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int i = 2 * q + t;
        if (i < grp.count) a.o[(size_t)hrow[i] * H + row] = ldexpf(acc[2 * (hr & 1) + t] * rw, sig[i]);
      }
    }
  }
}

}  // namespace moe
