// Expert-slot cache kernels: the ensure_experts remap with the LRU state on
// the device, the (a,b) precision-ladder classifier, and the grouping of
// (token, rank) pairs by expert.
//
// Sources: "Running DeepSeek-V4-Flash across four free GPUs", section "What
// the expert cache actually does" (in-place id -> slot remap, only misses
// copied, LRU, one cache global across layers) and section
// "moe_cache_size=128 is too small" (capacity floor); "An elephant through a
// straw", section "Not all six experts matter equally" (the ladder).
//
// One thread block of 1024 threads does a whole call; the work is a handful
// of block-wide passes over the call's entries, its distinct experts and the
// slots, all in shared memory:
//   1. first appearance of every expert (atomicMin of the flat entry index);
//   2. a bitmap of first-appearance positions and its prefix popcount give
//      every distinct expert its first-appearance order and give the longest
//      token prefix whose distinct experts fit the slots;
//   3. hits are looked up in key_to_slot; they are pinned by construction
//      (a slot is pinned iff its key is one of this call's distinct keys);
//   4. misses take empty slots by ascending index, then the unpinned slots
//      with the smallest stamps (rank counting in shared memory, or a binary
//      search over stamp values for very large candidate sets);
//   5. stamps become clock + first-appearance order.
#include <limits.h>

#include "common.cuh"

namespace moe {

constexpr int kEnsureThreads = 1024;
constexpr int kMaxEntries = 65536;

struct PassSmem {
  int* first_idx;    // [E]
  int* ord_of;       // [E]
  int* key_by_ord;   // [E]
  int* slot_of_ord;  // [E]
  int* mrank;        // [E]
  int* victims;      // [E]
  uint32_t* bitmap;  // [W]
  int* wprefix;      // [W]
  uint64_t* cand_stamp;  // [CMAX]
  int* cand_slot;        // [CMAX]
  int* ws;               // [34] scan workspace
  int* scal;             // [16] scalars
  unsigned long long* clock0;  // [1]
  int E, W, CMAX;
};

enum { SC_INVALID = 0, SC_DTOTAL, SC_NREL, SC_D, SC_M, SC_NEMPTY, SC_C };

__host__ __device__ inline size_t pass_smem_bytes(int E, int W, int CMAX) {
  return (size_t)6 * E * 4 + (size_t)W * 8 + (size_t)CMAX * 12 + 34 * 4 + 16 * 4 + 16;
}

__device__ PassSmem carve(uint8_t* base, int E, int W, int CMAX) {
  PassSmem s;
  uint8_t* p = base;
  s.cand_stamp = (uint64_t*)p;
  p += (size_t)CMAX * 8;
  s.clock0 = (unsigned long long*)p;
  p += 16;
  s.first_idx = (int*)p;
  p += E * 4;
  s.ord_of = (int*)p;
  p += E * 4;
  s.key_by_ord = (int*)p;
  p += E * 4;
  s.slot_of_ord = (int*)p;
  p += E * 4;
  s.mrank = (int*)p;
  p += E * 4;
  s.victims = (int*)p;
  p += E * 4;
  s.cand_slot = (int*)p;
  p += (size_t)CMAX * 4;
  s.bitmap = (uint32_t*)p;
  p += (size_t)W * 4;
  s.wprefix = (int*)p;
  p += (size_t)W * 4;
  s.ws = (int*)p;
  p += 34 * 4;
  s.scal = (int*)p;
  s.E = E;
  s.W = W;
  s.CMAX = CMAX;
  return s;
}

// Entries of a pass: tokens [tb, tend), ranks [lo, hi) of ids [T, k]; an
// entry is skipped when its id is negative or (skip_tags != null) its tag is
// MOE_TAG_FP4 (resolved by an earlier pass).
struct Entries {
  const int32_t* ids;
  const int8_t* skip_tags;
  int k, lo, hi, tb, tend;
  __device__ int R() const { return hi - lo; }
  __device__ int count() const { return (tend - tb) * (hi - lo); }
  __device__ size_t index(int f) const {
    const int r = hi - lo;
    return (size_t)(tb + f / r) * k + (lo + f % r);
  }
  __device__ int expert(int f) const {
    const size_t i = index(f);
    if (skip_tags && skip_tags[i] == MOE_TAG_FP4) return -1;
    return ids[i];
  }
};

__device__ __forceinline__ int count_first_below(const PassSmem& s, int p, int NE, int dtotal) {
  if (p >= NE) return dtotal;
  return s.wprefix[p >> 5] + __popc(s.bitmap[p >> 5] & ((1u << (p & 31)) - 1u));
}

// Steps 1-2: first appearance and first-appearance order of every distinct
// expert among the entries.  Returns the number of distinct experts (or -1
// if some id >= E).
__device__ int analyze(const PassSmem& s, const Entries& en) {
  const int tid = threadIdx.x, NT = blockDim.x;
  const int NE = en.count();
  const int W = (NE + 31) >> 5;
  __syncthreads();  // earlier readers of the shared arrays are done
  for (int e = tid; e < s.E; e += NT) {
    s.first_idx[e] = INT_MAX;
    s.ord_of[e] = INT_MAX;
  }
  for (int w = tid; w < W; w += NT) s.bitmap[w] = 0u;
  if (tid == 0) s.scal[SC_INVALID] = 0;
  __syncthreads();
  for (int f = tid; f < NE; f += NT) {
    const int e = en.expert(f);
    if (e >= s.E)
      s.scal[SC_INVALID] = 1;
    else if (e >= 0)
      atomicMin(&s.first_idx[e], f);
  }
  __syncthreads();
  if (s.scal[SC_INVALID]) return -1;
  for (int e = tid; e < s.E; e += NT) {
    const int fi = s.first_idx[e];
    if (fi != INT_MAX) atomicOr(&s.bitmap[fi >> 5], 1u << (fi & 31));
  }
  __syncthreads();
  const int wpt = (W + NT - 1) / NT;
  const int w0 = min(W, tid * wpt), w1 = min(W, w0 + wpt);
  int local = 0;
  for (int w = w0; w < w1; ++w) local += __popc(s.bitmap[w]);
  int total;
  int run = block_exclusive_scan(local, s.ws, &total);
  for (int w = w0; w < w1; ++w) {
    s.wprefix[w] = run;
    run += __popc(s.bitmap[w]);
  }
  __syncthreads();
  for (int e = tid; e < s.E; e += NT) {
    const int fi = s.first_idx[e];
    if (fi != INT_MAX) {
      const int o = s.wprefix[fi >> 5] + __popc(s.bitmap[fi >> 5] & ((1u << (fi & 31)) - 1u));
      s.ord_of[e] = o;
      s.key_by_ord[o] = e;
    }
  }
  __syncthreads();
  return total;
}

// Longest token prefix (relative count) whose distinct experts fit `cap`,
// after analyze().  Writes the distinct count of that prefix to *D.  Returns
// 0 when the first token alone does not fit.
__device__ int chunk_tokens(const PassSmem& s, const Entries& en, int dtotal, int cap, int* D) {
  const int n_all = en.tend - en.tb;
  if (dtotal <= cap) {
    *D = dtotal;
    return n_all;
  }
  const int fstar = s.first_idx[s.key_by_ord[cap]];
  const int n_rel = fstar / en.R();
  *D = count_first_below(s, n_rel * en.R(), en.count(), dtotal);
  return n_rel;
}

// Eviction order of an occupied slot among the candidates (smaller goes
// first): its stamp under LRU; under LFU the worth of its key (count halved
// once per epoch since it was written) above the stamp's low 44 bits, so equal
// worths fall back to the stamp order.
__device__ __forceinline__ uint64_t evict_order(const CacheDev& c, int slot, uint32_t epoch) {
  const uint64_t st = c.slot_stamp[slot];
  if (c.policy != MOE_EVICT_LFU) return st;
  const int key = c.slot_key[slot];
  const uint32_t sh = min(31u, epoch - c.freq_epoch[key]);
  return ((uint64_t)(c.freq[key] >> sh) << 44) | (st & ((1ull << 44) - 1));
}

// Steps 3-5 for the D distinct experts found by analyze(): resolve hits,
// place misses (FETCH), stamp.  Leaves the final slot (or -1) of every
// first-appearance order in slot_of_ord.  Returns the number of misses.
__device__ int resolve(const PassSmem& s, CacheDev c, int layer, int D, int mode,
                       int32_t* miss_key, int32_t* miss_slot) {
  const int tid = threadIdx.x, NT = blockDim.x;
  const int E = s.E;
  const bool lfu = c.policy == MOE_EVICT_LFU;
  const unsigned long long calls0 = lfu ? *c.calls : 0ull;  // read by all before thread 0 writes it back
  const uint32_t epoch = lfu ? (uint32_t)(calls0 / (unsigned long long)c.decay_calls) : 0u;
  if (tid == 0) *s.clock0 = *c.clock;
  for (int q = tid; q < D; q += NT) s.slot_of_ord[q] = c.key_to_slot[layer * E + s.key_by_ord[q]];
  __syncthreads();
  int M = 0;
  if (mode == MOE_FETCH) {
    // miss ranks in first-appearance order
    const int qpt = (D + NT - 1) / NT;
    const int q0 = min(D, tid * qpt), q1 = min(D, q0 + qpt);
    int local = 0;
    for (int q = q0; q < q1; ++q) local += s.slot_of_ord[q] < 0;
    int run = block_exclusive_scan(local, s.ws, &M);
    for (int q = q0; q < q1; ++q)
      if (s.slot_of_ord[q] < 0) s.mrank[q] = run++;
    if (M > 0) {
      // empty slots by ascending index
      const int S = c.S;
      const int spt = (S + NT - 1) / NT;
      const int s0 = min(S, tid * spt), s1 = min(S, s0 + spt);
      int ne = 0;
      for (int i = s0; i < s1; ++i) ne += c.slot_key[i] < 0;
      int n_empty;
      int r = block_exclusive_scan(ne, s.ws, &n_empty);
      for (int i = s0; i < s1 && r < M; ++i)
        if (c.slot_key[i] < 0) s.victims[r++] = i;
      const int take_empty = min(M, n_empty);
      const int r_lru = M - take_empty;
      if (r_lru > 0) {
        // candidates: occupied and not needed by this call
        int nc = 0;
        for (int i = s0; i < s1; ++i) {
          const int key = c.slot_key[i];
          const bool pinned = key >= 0 && key / E == layer && s.ord_of[key % E] < D;
          nc += (key >= 0 && !pinned);
        }
        int C;
        int cpos = block_exclusive_scan(nc, s.ws, &C);
        if (C <= s.CMAX) {
          for (int i = s0; i < s1; ++i) {
            const int key = c.slot_key[i];
            const bool pinned = key >= 0 && key / E == layer && s.ord_of[key % E] < D;
            if (key >= 0 && !pinned) {
              s.cand_stamp[cpos] = evict_order(c, i, epoch);
              s.cand_slot[cpos] = i;
              ++cpos;
            }
          }
        } else {
          // r_lru-th smallest stamp by binary search over stamp values, then
          // keep exactly the r_lru candidates at or below it (stamps are unique)
          unsigned long long lo = 0, hi = *s.clock0;
          if (lfu) hi |= (unsigned long long)kFreqCap << 44;
          while (lo < hi) {
            const unsigned long long mid = lo + (hi - lo) / 2;
            int cnt = 0;
            for (int i = s0; i < s1; ++i) {
              const int key = c.slot_key[i];
              const bool pinned = key >= 0 && key / E == layer && s.ord_of[key % E] < D;
              cnt += (key >= 0 && !pinned && evict_order(c, i, epoch) <= mid);
            }
            const int tot = block_sum(cnt, s.ws);
            if (tot >= r_lru)
              hi = mid;
            else
              lo = mid + 1;
          }
          int nk = 0;
          for (int i = s0; i < s1; ++i) {
            const int key = c.slot_key[i];
            const bool pinned = key >= 0 && key / E == layer && s.ord_of[key % E] < D;
            nk += (key >= 0 && !pinned && evict_order(c, i, epoch) <= lo);
          }
          int kpos = block_exclusive_scan(nk, s.ws, &C);
          for (int i = s0; i < s1; ++i) {
            const int key = c.slot_key[i];
            const bool pinned = key >= 0 && key / E == layer && s.ord_of[key % E] < D;
            if (key >= 0 && !pinned && evict_order(c, i, epoch) <= lo) {
              s.cand_stamp[kpos] = evict_order(c, i, epoch);
              s.cand_slot[kpos] = i;
              ++kpos;
            }
          }
        }
        __syncthreads();
        for (int i = tid; i < C; i += NT) {
          const uint64_t st = s.cand_stamp[i];
          int rank = 0;
          for (int j = 0; j < C; ++j) rank += s.cand_stamp[j] < st;
          if (rank < r_lru) s.victims[take_empty + rank] = s.cand_slot[i];
        }
      }
      __syncthreads();
      for (int q = tid; q < D; q += NT) {
        if (s.slot_of_ord[q] >= 0) continue;
        const int m = s.mrank[q];
        const int v = s.victims[m];
        const int key = layer * E + s.key_by_ord[q];
        const int old = c.slot_key[v];
        if (old >= 0) c.key_to_slot[old] = -1;
        c.slot_key[v] = key;
        c.key_to_slot[key] = v;
        s.slot_of_ord[q] = v;
        miss_key[m] = key;
        miss_slot[m] = v;
      }
      __syncthreads();
    }
  }
  const unsigned long long clk = *s.clock0;
  for (int q = tid; q < D; q += NT) {
    const int sl = s.slot_of_ord[q];
    if (sl >= 0) c.slot_stamp[sl] = clk + (unsigned long long)q;
    if (lfu) {
      // every distinct key of the call, resident or not: worth + 1, capped
      const int key = layer * E + s.key_by_ord[q];
      const uint32_t sh = min(31u, epoch - c.freq_epoch[key]);
      c.freq[key] = min((c.freq[key] >> sh) + 1u, kFreqCap);
      c.freq_epoch[key] = epoch;
    }
  }
  __syncthreads();
  if (tid == 0) {
    *c.clock = clk + (unsigned long long)D;
    if (lfu) *c.calls = calls0 + 1;
  }
  return M;
}

// Writes the resolved slot of every processed entry (and its tag when
// tags_out is given and the slot is valid).
__device__ void write_slots(const PassSmem& s, const Entries& en, int32_t* slots_out, int8_t* tags_out,
                            int8_t tag) {
  const int NE = en.count();
  for (int f = threadIdx.x; f < NE; f += blockDim.x) {
    const int e = en.expert(f);
    if (e < 0) continue;
    const size_t i = en.index(f);
    const int sl = s.slot_of_ord[s.ord_of[e]];
    slots_out[i] = sl;
    if (tags_out && sl >= 0) tags_out[i] = tag;
  }
}

__global__ void __launch_bounds__(kEnsureThreads)
    slot_ensure_kernel(CacheDev c, int layer, const int32_t* ids, int32_t* slots_out, int T, int k,
                       int lo, int hi, int mode, int tb, int32_t* miss_key, int32_t* miss_slot,
                       int32_t* miss_count, int32_t* tokens_done, int W, int CMAX) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  pdl_launch_dependents();  // the forward's plan may set up meanwhile
  pdl_wait();               // launched early behind the router
  PassSmem s = carve(smem_raw, c.E, W, CMAX);
  Entries en{ids, nullptr, k, lo, hi, tb, max(T, tb)};
  const bool mark_rest = mode == MOE_FETCH_MARK_REST;
  if (mark_rest) mode = MOE_FETCH;
  // MOE_FETCH_MARK_REST: entries of tokens [from, T) get slot -1.
  auto mark_from = [&](int from) {
    if (!mark_rest) return;
    Entries rest{ids, nullptr, k, lo, hi, from, en.tend};
    for (int f = threadIdx.x; f < rest.count(); f += blockDim.x)
      if (rest.expert(f) >= 0) slots_out[rest.index(f)] = -1;
  };
  const int dtotal = analyze(s, en);
  if (dtotal < 0) {
    mark_from(tb);
    if (threadIdx.x == 0) {
      *miss_count = -MOE_ERR_INVALID;
      *tokens_done = tb;
    }
    return;
  }
  int D = dtotal, n_rel = en.tend - en.tb;
  if (mode == MOE_FETCH) {
    n_rel = chunk_tokens(s, en, dtotal, c.S, &D);
    if (n_rel == 0 && en.tend > en.tb) {
      mark_from(tb);
      if (threadIdx.x == 0) {
        *miss_count = -MOE_ERR_CAPACITY;
        *tokens_done = tb;
      }
      return;
    }
  }
  const int M = resolve(s, c, layer, D, mode, miss_key, miss_slot);
  mark_from(tb + n_rel);
  en.tend = en.tb + n_rel;
  write_slots(s, en, slots_out, nullptr, 0);
  if (threadIdx.x == 0) {
    *miss_count = M;
    *tokens_done = tb + n_rel;
  }
}

// The ladder: all five passes of one chunk in one block.
__global__ void __launch_bounds__(kEnsureThreads)
    ladder_kernel(CacheDev c4, CacheDev c2, int layer, const int32_t* ids, const float* w, int T,
                  int k, int a, int b, int tb, int32_t* slots_out, int8_t* tags_out, float* w_out,
                  int32_t* mk4, int32_t* ms4, int32_t* mc4, int32_t* mk2, int32_t* ms2,
                  int32_t* mc2, int32_t* tokens_done, int W, int CMAX) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  PassSmem s = carve(smem_raw, c4.E, W, CMAX);
  const int tend_all = max(T, tb);
  auto fail_all = [&](int code) {
    if (threadIdx.x == 0) {
      *mc4 = -code;
      *mc2 = -code;
      *tokens_done = tb;
    }
  };
  // chunk: distinct rank-[0,a) experts fit the FP4 pool, rank-[a,b) the 2-bit pool
  Entries e1{ids, nullptr, k, 0, a, tb, tend_all};
  int dt = analyze(s, e1);
  if (dt < 0) return fail_all(MOE_ERR_INVALID);
  int D1;
  int n4 = chunk_tokens(s, e1, dt, c4.S, &D1);
  int n2 = tend_all - tb;
  if (b > a) {
    Entries e2{ids, nullptr, k, a, b, tb, tend_all};
    int dt2 = analyze(s, e2);
    if (dt2 < 0) return fail_all(MOE_ERR_INVALID);
    int D2;
    n2 = chunk_tokens(s, e2, dt2, c2.S, &D2);
  }
  const int n = min(n4, n2);
  if (n == 0 && tend_all > tb) return fail_all(MOE_ERR_CAPACITY);
  const int tend = tb + n;
  // every entry of the chunk starts dropped
  for (int f = threadIdx.x; f < n * k; f += blockDim.x) {
    const size_t i = (size_t)tb * k + f;
    slots_out[i] = -1;
    tags_out[i] = MOE_TAG_DROP;
  }
  __syncthreads();
  int M4 = 0, M2 = 0;
  {  // (i) FP4 FETCH, ranks [0, a)
    Entries en{ids, nullptr, k, 0, a, tb, tend};
    const int d = analyze(s, en);
    M4 = resolve(s, c4, layer, d, MOE_FETCH, mk4, ms4);
    write_slots(s, en, slots_out, tags_out, MOE_TAG_FP4);
    __syncthreads();
  }
  if (b > a) {  // (ii) FP4 LOOKUP then 2-bit FETCH, ranks [a, b)
    Entries en{ids, nullptr, k, a, b, tb, tend};
    int d = analyze(s, en);
    resolve(s, c4, layer, d, MOE_LOOKUP, nullptr, nullptr);
    write_slots(s, en, slots_out, tags_out, MOE_TAG_FP4);
    __syncthreads();
    Entries en2{ids, tags_out, k, a, b, tb, tend};
    d = analyze(s, en2);
    M2 = resolve(s, c2, layer, d, MOE_FETCH, mk2, ms2);
    write_slots(s, en2, slots_out, tags_out, MOE_TAG_INT2);
    __syncthreads();
  }
  if (k > b) {  // (iii) FP4 LOOKUP, then 2-bit LOOKUP, ranks [b, k); the rest stay dropped
    Entries en{ids, nullptr, k, b, k, tb, tend};
    int d = analyze(s, en);
    resolve(s, c4, layer, d, MOE_LOOKUP, nullptr, nullptr);
    write_slots(s, en, slots_out, tags_out, MOE_TAG_FP4);
    __syncthreads();
    Entries en2{ids, tags_out, k, b, k, tb, tend};
    d = analyze(s, en2);
    resolve(s, c2, layer, d, MOE_LOOKUP, nullptr, nullptr);
    write_slots(s, en2, slots_out, tags_out, MOE_TAG_INT2);
    __syncthreads();
  }
  // a 2-bit LOOKUP miss writes slot -1 with the tag left at DROP: keep it so
  for (int t = tb + threadIdx.x; t < tend; t += blockDim.x) {
    float sum = 0.f;
    for (int j = 0; j < k; ++j) {
      const size_t i = (size_t)t * k + j;
      if (tags_out[i] == MOE_TAG_DROP) slots_out[i] = -1;
      else sum += w[i];
    }
    for (int j = 0; j < k; ++j) {
      const size_t i = (size_t)t * k + j;
      w_out[i] = tags_out[i] == MOE_TAG_DROP ? 0.f : w[i] / sum;
    }
  }
  if (threadIdx.x == 0) {
    *mc4 = M4;
    *mc2 = M2;
    *tokens_done = tend;
  }
}

// Stable grouping of pairs by expert: one block; histogram, scan, then the
// pairs are placed tile by tile with the warps of a tile taking turns, so the
// order within an expert is the pair order.
__global__ void __launch_bounds__(1024)
    group_pairs_kernel(const int32_t* ids, int P, int E, int32_t* offsets, int32_t* perm,
                       int32_t* err) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  int* cnt = (int*)smem_raw;  // [E]
  int* ws = cnt + E;          // [34]
  int* bad = ws + 34;
  const int tid = threadIdx.x, NT = blockDim.x, lane = tid & 31, wid = tid >> 5;
  for (int e = tid; e < E; e += NT) cnt[e] = 0;
  if (tid == 0) *bad = 0;
  __syncthreads();
  for (int p = tid; p < P; p += NT) {
    const int e = ids[p];
    if (e >= E) *bad = 1;
    else if (e >= 0) atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  const int ept = (E + NT - 1) / NT;
  const int e0 = min(E, tid * ept), e1 = min(E, e0 + ept);
  int local = 0;
  for (int e = e0; e < e1; ++e) local += cnt[e];
  int total;
  int run = block_exclusive_scan(local, ws, &total);
  for (int e = e0; e < e1; ++e) {
    const int c = cnt[e];
    cnt[e] = run;
    offsets[e] = run;
    run += c;
  }
  if (tid == 0) {
    offsets[E] = total;
    *err = *bad ? MOE_ERR_INVALID : 0;
  }
  __syncthreads();
  const int nwarps = NT >> 5;
  for (int base = 0; base < P; base += NT) {
    const int p = base + tid;
    const int e = (p < P) ? ids[p] : -1;
    const bool valid = e >= 0 && e < E;
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const bool leader = rank == 0;
    for (int w = 0; w < nwarps; ++w) {
      if (wid == w && valid) {
        perm[cnt[e] + rank] = p;
        __syncwarp(peers);
        if (leader) cnt[e] += __popc(peers);
      }
      __syncthreads();
    }
  }
}

// Multi-block form of the same stable grouping for large pair counts: each
// block owns a contiguous segment of kSeg pairs.  (1) per-segment histograms;
// (2) one block turns them into per-(segment, expert) start positions, ordered
// expert-major then segment; (3) each segment places its pairs in order, the
// warps of a tile taking turns, so the order within an expert is pair order.
constexpr int kSeg = 1024;

__global__ void __launch_bounds__(1024) group_hist_kernel(const int32_t* ids, int P, int E, int* cnt, int32_t* err) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  int* h = (int*)smem_raw;
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
  const int p0 = blockIdx.x * kSeg, p1 = min(P, p0 + kSeg);
  for (int p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    const int e = ids[p];
    if (e >= E) atomicExch(err, MOE_ERR_INVALID);
    else if (e >= 0) atomicAdd(&h[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[(size_t)blockIdx.x * E + e] = h[e];
}

__global__ void __launch_bounds__(1024) group_scan_kernel(int nb, int E, int* cnt, int32_t* offsets) {
  __shared__ int ws[34];
  const int tid = threadIdx.x, NT = blockDim.x;
  const int ept = (E + NT - 1) / NT;
  const int e0 = min(E, tid * ept), e1 = min(E, e0 + ept);
  int local = 0;
  for (int e = e0; e < e1; ++e)
    for (int b = 0; b < nb; ++b) local += cnt[(size_t)b * E + e];
  int total;
  int run = block_exclusive_scan(local, ws, &total);
  for (int e = e0; e < e1; ++e) {
    offsets[e] = run;
    for (int b = 0; b < nb; ++b) {
      const int c = cnt[(size_t)b * E + e];
      cnt[(size_t)b * E + e] = run;
      run += c;
    }
  }
  if (tid == 0) offsets[E] = total;
}

__global__ void __launch_bounds__(1024) group_place_kernel(const int32_t* ids, int P, int E, const int* cnt,
                                                           int32_t* perm) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  int* off = (int*)smem_raw;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nwarps = blockDim.x >> 5;
  for (int e = tid; e < E; e += blockDim.x) off[e] = cnt[(size_t)blockIdx.x * E + e];
  __syncthreads();
  const int p0 = blockIdx.x * kSeg, p1 = min(P, p0 + kSeg);
  for (int base = p0; base < p1; base += blockDim.x) {
    const int p = base + tid;
    const int e = (p < p1) ? ids[p] : -1;
    const bool valid = e >= 0 && e < E;
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    for (int w = 0; w < nwarps; ++w) {
      if (wid == w && valid) {
        perm[off[e] + rank] = p;
        __syncwarp(peers);
        if (rank == 0) off[e] += __popc(peers);
      }
      __syncthreads();
    }
  }
}

moe_status group_pairs_multi(const int32_t* ids, int P, int E, int32_t* offsets, int32_t* perm, int32_t* d_error,
                             int* cnt_ws, cudaStream_t stream) {
  const int nb = (P + kSeg - 1) / kSeg;
  const size_t smem = (size_t)E * 4;
  if (smem > 48 * 1024) {
    cudaError_t e1 = cudaFuncSetAttribute(group_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    cudaError_t e2 = cudaFuncSetAttribute(group_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e1 != cudaSuccess) return cuda_fail(e1, "cudaFuncSetAttribute(group_hist_kernel)");
    if (e2 != cudaSuccess) return cuda_fail(e2, "cudaFuncSetAttribute(group_place_kernel)");
  }
  ProfScope ps(MOE_K_GROUP, stream);
  // d_error is cleared by the calling entry point, once per call
  if (nb > 0) group_hist_kernel<<<nb, 1024, smem, stream>>>(ids, P, E, cnt_ws, d_error);
  group_scan_kernel<<<1, 1024, 0, stream>>>(nb, E, cnt_ws, offsets);
  if (nb > 0) group_place_kernel<<<nb, 1024, smem, stream>>>(ids, P, E, cnt_ws, perm);
  return check_launch("group_pairs_multi");
}

size_t group_pairs_multi_ws(int P, int E) { return (size_t)((P + kSeg - 1) / kSeg) * E * 4; }

static moe_status prepare_smem(const void* kernel, size_t bytes) {
  static_assert(sizeof(int) == 4, "int");
  if (bytes > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic shared memory)");
  }
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_slot_ensure(moe_cache* cache, int layer_id, const int32_t* ids,
                                      int32_t* slots_out, int T, int k, int rank_lo, int rank_hi,
                                      int mode, int token_begin, int32_t* d_miss_key,
                                      int32_t* d_miss_slot, int32_t* d_miss_count,
                                      int32_t* d_tokens_done, cudaStream_t stream) {
  clear_error();
  MOE_ARG(cache != nullptr, "cache is null");
  MOE_ARG(layer_id >= 0 && layer_id < cache->L, "layer_id %d out of [0, %d)", layer_id, cache->L);
  MOE_ARG(T >= 0 && k >= 1 && k <= 64, "need T >= 0 and 1 <= k <= 64");
  MOE_ARG(0 <= rank_lo && rank_lo <= rank_hi && rank_hi <= k, "bad rank range [%d, %d)", rank_lo, rank_hi);
  MOE_ARG(mode == MOE_FETCH || mode == MOE_LOOKUP || mode == MOE_FETCH_MARK_REST, "bad mode");
  MOE_ARG(mode != MOE_FETCH_MARK_REST || (const void*)ids != (const void*)slots_out,
          "MOE_FETCH_MARK_REST needs slots_out separate from ids");
  MOE_ARG(token_begin >= 0, "token_begin < 0");
  MOE_ARG(ids && slots_out && d_miss_count && d_tokens_done, "null pointer");
  MOE_ARG(mode == MOE_LOOKUP || (d_miss_key && d_miss_slot), "FETCH needs miss lists");
  const long long NE = (long long)(T > token_begin ? T - token_begin : 0) * (rank_hi - rank_lo);
  MOE_ARG(NE <= kMaxEntries, "(T - token_begin) * (rank_hi - rank_lo) = %lld exceeds %d", NE, kMaxEntries);
  const int W = (int)((NE + 31) / 32) + 1;
  const int CMAX = cache->E > 1024 ? cache->E : 1024;
  const size_t smem = pass_smem_bytes(cache->E, W, CMAX);
  moe_status st = prepare_smem((const void*)slot_ensure_kernel, smem);
  if (st != MOE_OK) return st;
  ProfScope ps(MOE_K_ENSURE, stream);
  cudaError_t e = launch_pdl(slot_ensure_kernel, dim3(1), dim3(kEnsureThreads), smem, stream, cache->dev, layer_id,
                             ids, slots_out, T, k, rank_lo, rank_hi, mode, token_begin,
                             d_miss_key ? d_miss_key : d_miss_count, d_miss_slot ? d_miss_slot : d_miss_count,
                             d_miss_count, d_tokens_done, W, CMAX);
  if (e != cudaSuccess) return cuda_fail(e, "slot_ensure_kernel");
  return check_launch("slot_ensure_kernel");
}

extern "C" moe_status moe_ladder_classify(moe_cache* c4, moe_cache* c2, int layer_id, const int32_t* ids,
                                          const float* w, int T, int k, int a, int b, int token_begin,
                                          int32_t* slots_out, int8_t* tags_out, float* w_out,
                                          int32_t* mk4, int32_t* ms4, int32_t* mc4, int32_t* mk2,
                                          int32_t* ms2, int32_t* mc2, int32_t* tokens_done,
                                          cudaStream_t stream) {
  clear_error();
  MOE_ARG(c4 && c2, "cache is null");
  MOE_ARG(c4->E == c2->E && c4->L == c2->L, "the two caches must have the same L and E");
  MOE_ARG(c4->dev.policy == MOE_EVICT_LRU && c2->dev.policy == MOE_EVICT_LRU, "the ladder needs LRU caches");
  MOE_ARG(layer_id >= 0 && layer_id < c4->L, "layer_id out of range");
  MOE_ARG(T >= 0 && k >= 1 && k <= 64, "need T >= 0 and 1 <= k <= 64");
  MOE_ARG(1 <= a && a <= b && b <= k, "need 1 <= a <= b <= k");
  MOE_ARG(token_begin >= 0, "token_begin < 0");
  MOE_ARG(ids && w && slots_out && tags_out && w_out && mk4 && ms4 && mc4 && mk2 && ms2 && mc2 &&
              tokens_done,
          "null pointer");
  MOE_ARG((const void*)ids != (const void*)slots_out, "slots_out must not alias ids");
  const long long NE = (long long)(T > token_begin ? T - token_begin : 0) * k;
  MOE_ARG(NE <= kMaxEntries, "(T - token_begin) * k exceeds %d", kMaxEntries);
  const int W = (int)((NE + 31) / 32) + 1;
  const int CMAX = c4->E > 1024 ? c4->E : 1024;
  const size_t smem = pass_smem_bytes(c4->E, W, CMAX);
  moe_status st = prepare_smem((const void*)ladder_kernel, smem);
  if (st != MOE_OK) return st;
  ProfScope ps(MOE_K_LADDER, stream);
  ladder_kernel<<<1, kEnsureThreads, smem, stream>>>(c4->dev, c2->dev, layer_id, ids, w, T, k, a, b,
                                                     token_begin, slots_out, tags_out, w_out, mk4, ms4,
                                                     mc4, mk2, ms2, mc2, tokens_done, W, CMAX);
  return check_launch("ladder_kernel");
}

extern "C" moe_status moe_group_pairs(const int32_t* ids, int T, int k, int E, int32_t* offsets,
                                      int32_t* perm, int32_t* d_error, cudaStream_t stream) {
  clear_error();
  MOE_ARG(T >= 0 && k >= 1 && E >= 1 && E <= 16384, "need T >= 0, k >= 1, 1 <= E <= 16384");
  MOE_ARG(offsets && d_error && (T == 0 || (ids && perm)), "null pointer");
  MOE_ARG((long long)T * k < (1LL << 31), "too many pairs");
  const size_t smem = (size_t)E * 4 + 36 * 4;
  moe_status st = prepare_smem((const void*)group_pairs_kernel, smem);
  if (st != MOE_OK) return st;
  ProfScope ps(MOE_K_GROUP, stream);
  group_pairs_kernel<<<1, 1024, smem, stream>>>(ids, T * k, E, offsets, perm, d_error);
  return check_launch("group_pairs_kernel");
}
