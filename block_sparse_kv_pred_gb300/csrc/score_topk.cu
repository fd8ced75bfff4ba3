// scout_score_topk: digest scoring, per-unit top-k, residency split, CPU work list.
// ScoutAttention (arXiv HTML), section 3.2 and Algorithm 1: B_pred = TopK(q K_digest^T),
// B_cpu = B_pred \ B_gpu.
//
// One persistent, warp-specialised kernel (one CTA per SM):
//  * warp 12 streams work items (unit, 128-row digest chunk) with TMA: four 128-byte
//    swizzled boxes of the chunk plus the unit's query rows, into a ring of stages;
//  * warps 0..7 score one 16-row tile of each chunk on the tensor cores.  A score is a
//    dot product over the 256 [min | max] digest values (q- pairs with min, q+ with
//    max) or over the 128 fp32 means split exactly into three bf16 terms, so mma.sync
//    with bf16 operands and fp32 accumulation computes it (products are exact).  The
//    score pooled over the unit's G query heads (maximum) becomes an orderable key in
//    shared memory;
//  * warps 8..11 select each unit as soon as its chunks are scored: radix select of the
//    k-th key, then one ordered compaction into top-k, resident, CPU and delta lists.
// CTA c owns the contiguous item range [c I / Gp, (c+1) I / Gp), so almost every unit
// is scored and selected inside one CTA; a unit cut by a range boundary goes through
// global memory and is selected by whichever of its CTAs adds its last chunks to a
// per-unit counter.
#include <mutex>

#include "common.cuh"

namespace scout {
namespace {

constexpr int kScoreWarps = 8;
constexpr int kSelWarps = 4;
constexpr int kSelThreads = kSelWarps * 32;
constexpr int kProducer = kScoreWarps + kSelWarps;  // warp index of the TMA producer
constexpr int kThreadsAll = (kProducer + 1) * 32;
constexpr int kChunk = kScoreWarps * 16;  // digest rows (blocks) per work item
constexpr int kBoxBytes = kChunk * 128;   // one 128-row x 128-byte TMA box
constexpr int kMaxStagesT = 3;

__device__ __forceinline__ uint32_t trunc_bf16(float x) { return __float_as_uint(x) & 0xFFFF0000u; }

// Orderable key of an fp32 score: larger score -> larger key; -0 and +0 equal.
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t b = __float_as_uint(s == 0.f ? 0.f : s);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The query group sits in shared memory with rows kQStride bf16 apart (272 bytes):
// the 8 rows a fragment load touches then fall on distinct banks.
constexpr int kQStride = kD + 8;
constexpr int kQBytes = kMaxG * kQStride * 2;
// digest chunk + the unit's query group, rounded so every stage starts 1024-aligned
constexpr int kStageBytesT = (4 * kBoxBytes + kQBytes + 1023) / 1024 * 1024;

// Keep the bf16 halves of a pair whose sign bit is clear (q+) or set (q-).
__device__ __forceinline__ uint32_t pos_part(uint32_t v) { return v & ~(((v >> 15) & 0x00010001u) * 0xFFFFu); }
__device__ __forceinline__ uint32_t neg_part(uint32_t v) { return v & (((v >> 15) & 0x00010001u) * 0xFFFFu); }

// q fragment (B operand) for the min/max kind, standard k order: k-step s covers
// digest values [16 s, 16 s + 16) of the [min | max] row, i.e. part s / 8 (min pairs
// with q-, max with q+) and channels (s % 8) * 16 + {2t, 2t+1, 2t+8, 2t+9}.
__device__ __forceinline__ void minmax_b_frag(const __nv_bfloat16* qs, int G, int lane, uint32_t (&bf)[16][2]) {
  const int g = lane >> 2, t = lane & 3;
  const uint32_t* row = reinterpret_cast<const uint32_t*>(qs + g * kQStride);
#pragma unroll
  for (int s8 = 0; s8 < 8; ++s8) {
    const uint32_t lo = g < G ? row[s8 * 8 + t] : 0u, hi = g < G ? row[s8 * 8 + t + 4] : 0u;
    bf[s8][0] = neg_part(lo);
    bf[s8][1] = neg_part(hi);
    bf[s8 + 8][0] = pos_part(lo);
    bf[s8 + 8][1] = pos_part(hi);
  }
}

// q fragment for the mean kind: load i of lane t covers channels i*16 + t*4 + {0..3}.
__device__ __forceinline__ void mean_b_frag(const __nv_bfloat16* qs, int G, int lane, uint32_t (&bf)[8][2]) {
  const int g = lane >> 2, t = lane & 3;
  const uint32_t* row = reinterpret_cast<const uint32_t*>(qs + g * kQStride);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    bf[i][0] = g < G ? row[i * 8 + 2 * t] : 0u;
    bf[i][1] = g < G ? row[i * 8 + 2 * t + 1] : 0u;
  }
}

// A chunk of 128 digest rows sits in shared memory as four TMA boxes of
// 128 rows x 128 bytes (row bytes [128 b, 128 b + 128) in box b), each with the
// 128-byte swizzle: 16-byte chunk c of row r lives at chunk c ^ (r % 8).
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int r, int C) {
  return base + (uint32_t)((C >> 3) * kBoxBytes + r * 128 + (((C & 7) ^ (r & 7)) << 4));
}

// Scores of the warp's 16 rows (local rows r0 .. r0 + 15): c = rows g, g + 8 x heads 2t, 2t+1.
template <int KIND>
__device__ __forceinline__ void score_tile(uint32_t tbase, int r0, int lane, const uint32_t (&bmm)[16][2],
                                           const uint32_t (&bme)[8][2], float (&c)[4]) {
  float acc[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  if (KIND == SCOUT_DIGEST_MINMAX) {
    const int r = r0 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
    for (int s = 0; s < 16; ++s) {  // four independent accumulation chains
      uint32_t a0, a1, a2, a3;
      ldsm_x4(tile_addr(tbase, r, 2 * s + (lane >> 4)), a0, a1, a2, a3);
      mma_bf16(acc[s & 3], a0, a1, a2, a3, bmm[s][0], bmm[s][1]);
    }
  } else {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // four fp32 channels i*16 + 4t .. +3 of rows g and g + 8, split exactly as hi + mid + lo (bf16)
      uint4 v0, v1;
      const uint32_t p0 = tile_addr(tbase, r0 + g, i * 4 + t), p1 = tile_addr(tbase, r0 + g + 8, i * 4 + t);
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v0.x), "=r"(v0.y), "=r"(v0.z), "=r"(v0.w) : "r"(p0));
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v1.x), "=r"(v1.y), "=r"(v1.z), "=r"(v1.w) : "r"(p1));
      const float x0[4] = {__uint_as_float(v0.x), __uint_as_float(v0.y), __uint_as_float(v0.z), __uint_as_float(v0.w)};
      const float x1[4] = {__uint_as_float(v1.x), __uint_as_float(v1.y), __uint_as_float(v1.z), __uint_as_float(v1.w)};
      float r0v[4], r1v[4];
      uint32_t h0[4], h1[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        h0[e] = trunc_bf16(x0[e]);
        h1[e] = trunc_bf16(x1[e]);
        r0v[e] = x0[e] - __uint_as_float(h0[e]);
        r1v[e] = x1[e] - __uint_as_float(h1[e]);
      }
#pragma unroll
      for (int part = 0; part < 3; ++part) {
        uint32_t a0[4], a1[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (part == 0) {
            a0[e] = h0[e];
            a1[e] = h1[e];
          } else if (part == 1) {
            a0[e] = trunc_bf16(r0v[e]);
            a1[e] = trunc_bf16(r1v[e]);
          } else {
            a0[e] = trunc_bf16(r0v[e] - __uint_as_float(trunc_bf16(r0v[e])));
            a1[e] = trunc_bf16(r1v[e] - __uint_as_float(trunc_bf16(r1v[e])));
          }
        }
        // pack two bf16 (upper halves of the fp32 patterns): low half = lower k
        const uint32_t A0 = (a0[0] >> 16) | a0[1], A1 = (a1[0] >> 16) | a1[1];
        const uint32_t A2 = (a0[2] >> 16) | a0[3], A3 = (a1[2] >> 16) | a1[3];
        mma_bf16(acc[part], A0, A1, A2, A3, bme[i][0], bme[i][1]);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) c[e] = (acc[0][e] + acc[1][e]) + (acc[2][e] + acc[3][e]);
}

struct TopkArgs {
  const __nv_bfloat16* q;
  const uint8_t* digest;
  const int32_t* seq_len;
  const uint32_t* resident_bits;
  const int32_t* prev_list;
  const int32_t* prev_count;
  int Hq, Hkv, G, P, nblk_cap, k, words, nchunk, stages;
  int user_scores;  // 1: the caller asked for every pooled score in `scores`
  int64_t n_items;
  float* scores;  // user buffer or workspace
  int32_t* counters;
  int32_t* status;
  int32_t *topk_idx, *topk_count, *res_list, *res_count, *cpu_list, *cpu_count, *delta_list, *delta_count;
};

__host__ __device__ constexpr int align4(int n) { return (n + 3) / 4 * 4; }  // words to a 16-byte multiple

__device__ __forceinline__ int unit_nvalid(const TopkArgs& a, int b) {
  return min(a.nblk_cap, (max(a.seq_len[b], 0) + a.P - 1) / a.P);
}

// The selector warps synchronise among themselves on named barrier 2.
__device__ __forceinline__ void sbar() { asm volatile("bar.sync 2, %0;" ::"n"(kSelThreads) : "memory"); }

// Exclusive prefix over the selector threads of four counters per thread; returns the totals.
__device__ __forceinline__ int4 sel_excl_scan4(int4 v, int4* wsum, int4& total) {
  const int lane = threadIdx.x & 31, w = (threadIdx.x >> 5) - kScoreWarps;
  int4 inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, inc.x, o), y = __shfl_up_sync(0xffffffffu, inc.y, o);
    const int z = __shfl_up_sync(0xffffffffu, inc.z, o), ww = __shfl_up_sync(0xffffffffu, inc.w, o);
    if (lane >= o) {
      inc.x += x;
      inc.y += y;
      inc.z += z;
      inc.w += ww;
    }
  }
  if (lane == 31) wsum[w] = inc;
  sbar();
  int4 base = make_int4(0, 0, 0, 0), tot = make_int4(0, 0, 0, 0);
#pragma unroll
  for (int i = 0; i < kSelWarps; ++i) {
    const int4 s = wsum[i];
    if (i < w) {
      base.x += s.x;
      base.y += s.y;
      base.z += s.z;
      base.w += s.w;
    }
    tot.x += s.x;
    tot.y += s.y;
    tot.z += s.z;
    tot.w += s.w;
  }
  sbar();
  total = tot;
  return make_int4(base.x + inc.x - v.x, base.y + inc.y - v.y, base.z + inc.z - v.z, base.w + inc.w - v.w);
}

constexpr int kDigitBits = 12;  // radix digit width of the selection
constexpr int kBins = 1 << kDigitBits;

struct SelShared {
  uint32_t* rbits;  // [words] residency of the unit
  uint32_t* pbits;  // [words] previous CPU list of the unit
  int* hist;        // [kBins]
  int4 wsum[kSelWarps];
  uint32_t kmin[kSelWarps], kmax[kSelWarps];
  int digit, remaining, count, nvalid;
};

// Loads the unit's residency bits and previous CPU list into shared memory; issued
// before the unit's keys are ready so the global-memory latency overlaps the scoring.
__device__ void prefetch_unit(const TopkArgs& a, int u, SelShared& ss) {
  const int st = threadIdx.x - kScoreWarps * 32;
  if (st == 0) ss.nvalid = unit_nvalid(a, u / a.Hkv);
  for (int i = st; i < a.words; i += kSelThreads) {
    ss.rbits[i] = a.resident_bits[(int64_t)u * a.words + i];
    ss.pbits[i] = 0u;
  }
  sbar();
  if (a.prev_list != nullptr) {
    const int pc = min(max(a.prev_count[u], 0), a.k);
    for (int i = st; i < pc; i += kSelThreads) {
      const int j = a.prev_list[(int64_t)u * a.k + i];
      if (j >= 0 && j < a.nblk_cap) atomicOr(&ss.pbits[j >> 5], 1u << (j & 31));
    }
  }
  sbar();
}

// Top-k of one unit's keys (in shared memory), split by residency, delta against the
// previous CPU list, ordered compaction.  Run by the 128 selector threads after
// prefetch_unit(u).
__device__ void select_unit(const TopkArgs& a, int u, const uint32_t* keys, SelShared& ss) {
  const int st = threadIdx.x - kScoreWarps * 32;  // 0 .. 127
  const int lane = threadIdx.x & 31, w = st >> 5;
  const int nvalid = ss.nvalid;
  const int keff = min(a.k, nvalid);
  uint32_t prefix = 0u, mask = 0u;
  int remaining = keff, count = nvalid;
  if (keff < nvalid) {
    // the leading bits every key shares need no radix pass
    uint32_t lo = 0xffffffffu, hi = 0u;
    for (int j = st; j < nvalid; j += kSelThreads) {
      lo = min(lo, keys[j]);
      hi = max(hi, keys[j]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
      ss.kmin[w] = lo;
      ss.kmax[w] = hi;
    }
    sbar();
#pragma unroll
    for (int i = 0; i < kSelWarps; ++i) {
      lo = min(lo, ss.kmin[i]);
      hi = max(hi, ss.kmax[i]);
    }
    int fixed = (lo == hi) ? 32 : __clz(lo ^ hi);  // leading bits common to all keys
    mask = fixed == 0 ? 0u : (fixed == 32 ? 0xffffffffu : ~(0xffffffffu >> fixed));
    prefix = lo & mask;
    // radix select on 12-bit digits below the common bits; it stops once the keys
    // sharing the current prefix are exactly the ones still needed
    while (fixed < 32 && remaining != count) {
      const int width = min(kDigitBits, 32 - fixed), shift = 32 - fixed - width;
      const uint32_t dmask = (1u << width) - 1u;
      for (int i = st; i < kBins / 4; i += kSelThreads) reinterpret_cast<int4*>(ss.hist)[i] = make_int4(0, 0, 0, 0);
      sbar();
      for (int j = st; j < nvalid; j += kSelThreads) {
        const uint32_t key = keys[j];
        if ((key & mask) == prefix) atomicAdd(&ss.hist[(key >> shift) & dmask], 1);
      }
      sbar();
      // thread st owns the 32 bins [kBins - 32 (st + 1), kBins - 32 st): high bins first
      constexpr int kPer = kBins / kSelThreads;
      const int top = kBins - kPer * st - 1;
      int sum = 0;
#pragma unroll 8
      for (int e = 0; e < kPer; ++e) sum += ss.hist[top - ((e + lane) & (kPer - 1))];  // rotated: no bank conflicts
      int4 tot4;
      const int before = sel_excl_scan4(make_int4(sum, 0, 0, 0), ss.wsum, tot4).x;
      if (before < remaining && remaining <= before + sum) {
        int acc = before;
        for (int e = 0; e < kPer; ++e) {
          const int c = ss.hist[top - e];
          if (acc < remaining && remaining <= acc + c) {
            ss.digit = top - e;
            ss.remaining = remaining - acc;
            ss.count = c;
            break;
          }
          acc += c;
        }
      }
      sbar();
      prefix |= (uint32_t)ss.digit << shift;
      mask |= dmask << shift;
      remaining = ss.remaining;
      count = ss.count;
      fixed += width;
    }
  }
  // selected: masked key above the prefix, or equal to it and (all equal ones needed,
  // or among the lowest-index `remaining` of them).  Thread st owns the contiguous
  // blocks [st per, st per + per) in groups of 8 (one residency byte, two 16-byte key
  // loads); per-thread counts are scanned once, so the lists come out in ascending
  // block order.
  const bool all_eq = remaining == count;
  const int per = ((nvalid + kSelThreads - 1) / kSelThreads + 7) / 8 * 8;
  const int jlo = min(nvalid, st * per), jhi = min(nvalid, jlo + per);
  int4 tot;
  int eq_base = 0;
  if (!all_eq) {
    int n_eq = 0;
    for (int j = jlo; j < jhi; ++j) n_eq += (keys[j] & mask) == prefix;
    eq_base = sel_excl_scan4(make_int4(n_eq, 0, 0, 0), ss.wsum, tot).x;
  }
  // pass 1: counts
  int4 cnt = make_int4(0, 0, 0, 0);
  int eqr = eq_base;
  for (int g0 = jlo; g0 < jhi; g0 += 8) {
    uint32_t kv[8];
    if (g0 + 8 <= jhi) {
      const uint4 x = *reinterpret_cast<const uint4*>(keys + g0), y = *reinterpret_cast<const uint4*>(keys + g0 + 4);
      kv[0] = x.x; kv[1] = x.y; kv[2] = x.z; kv[3] = x.w; kv[4] = y.x; kv[5] = y.y; kv[6] = y.z; kv[7] = y.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) kv[e] = g0 + e < jhi ? keys[g0 + e] : 0u;
    }
    const uint32_t rb = ss.rbits[g0 >> 5] >> (g0 & 31), pb = ss.pbits[g0 >> 5] >> (g0 & 31);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t mk = kv[e] & mask;
      const bool in = g0 + e < jhi, eq = in && mk == prefix;
      const bool sel = in && (mk > prefix || (eq && (all_eq || eqr < remaining)));
      eqr += eq;
      if (sel) {
        cnt.x += 1;
        if ((rb >> e) & 1u) cnt.y += 1;
        else {
          cnt.z += 1;
          cnt.w += ((pb >> e) & 1u) ? 0 : 1;
        }
      }
    }
  }
  int4 pos = sel_excl_scan4(cnt, ss.wsum, tot);
  // pass 2: writes
  const int64_t lb = (int64_t)u * a.k;
  eqr = eq_base;
  for (int g0 = jlo; g0 < jhi; g0 += 8) {
    uint32_t kv[8];
    if (g0 + 8 <= jhi) {
      const uint4 x = *reinterpret_cast<const uint4*>(keys + g0), y = *reinterpret_cast<const uint4*>(keys + g0 + 4);
      kv[0] = x.x; kv[1] = x.y; kv[2] = x.z; kv[3] = x.w; kv[4] = y.x; kv[5] = y.y; kv[6] = y.z; kv[7] = y.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) kv[e] = g0 + e < jhi ? keys[g0 + e] : 0u;
    }
    const uint32_t rb = ss.rbits[g0 >> 5] >> (g0 & 31), pb = ss.pbits[g0 >> 5] >> (g0 & 31);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t mk = kv[e] & mask;
      const bool in = g0 + e < jhi, eq = in && mk == prefix;
      const bool sel = in && (mk > prefix || (eq && (all_eq || eqr < remaining)));
      eqr += eq;
      if (sel) {
        const int j = g0 + e;
        a.topk_idx[lb + pos.x++] = j;
        if ((rb >> e) & 1u) {
          a.res_list[lb + pos.y++] = j;
        } else {
          a.cpu_list[lb + pos.z++] = j;
          if (!((pb >> e) & 1u)) a.delta_list[lb + pos.w++] = j;
        }
      }
    }
  }
  for (int i = st; i < a.k; i += kSelThreads) {
    if (i >= tot.x) a.topk_idx[lb + i] = -1;
    if (i >= tot.y) a.res_list[lb + i] = -1;
    if (i >= tot.z) a.cpu_list[lb + i] = -1;
    if (i >= tot.w) a.delta_list[lb + i] = -1;
  }
  if (st == 0) {
    a.topk_count[u] = tot.x;
    a.res_count[u] = tot.y;
    a.cpu_count[u] = tot.z;
    a.delta_count[u] = tot.w;
  }
  sbar();  // keys and scratch are reused by the next selection
}

template <int KIND>
__global__ void __launch_bounds__(kThreadsAll, 1) score_topk_kernel(const __grid_constant__ CUtensorMap tmD,
                                                                    const TopkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kMaxStagesT], empty_bar[kMaxStagesT], kfull[2], kempty[2];
  __shared__ SelShared ss;
  __shared__ int s_flag;
  // dynamic shared memory: [ring (1024-aligned)][2 key buffers][residency bits][previous-list bits]
  // [radix histogram]
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint32_t* keybuf = reinterpret_cast<uint32_t*>(ring + a.stages * kStageBytesT);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int i = 0; i < a.stages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kScoreWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kfull[i], kScoreWarps);
      mbar_init(&kempty[i], 1);
    }
    fence_mbar_init();
    // every region starts 16-byte aligned (the histogram is zeroed with int4 stores)
    ss.rbits = keybuf + 2 * align4(a.nblk_cap);
    ss.pbits = ss.rbits + align4(a.words);
    ss.hist = reinterpret_cast<int*>(ss.pbits + align4(a.words));
  }
  __syncthreads();
  const int64_t Gp = gridDim.x;  // the host launches at most one CTA per item
  const int64_t it0 = blockIdx.x * a.n_items / Gp, it1 = (blockIdx.x + 1) * a.n_items / Gp;
  const int u_first = (int)(it0 / a.nchunk), u_last = (int)((it1 - 1) / a.nchunk);

  if (warp == kProducer) {
    // ---------------- producer warp ------------------------------------------
    if (lane != 0) return;
    prefetch_tmap(&tmD);
    int64_t issued = 0;
    for (int64_t i = 0; i < it1 - it0; ++i) {
      const int64_t item = it0 + i;
      const int u = (int)(item / a.nchunk), ch = (int)(item - (int64_t)u * a.nchunk);
      const int b = u / a.Hkv, kvh = u - b * a.Hkv;
      const int st = (int)(i % a.stages);
      if (!mbar_wait(&empty_bar[st], (uint32_t)((i / a.stages) & 1) ^ 1u)) {
        report(a.status, SCOUT_DEV_TIMEOUT);
        break;
      }
      uint8_t* sp = ring + st * kStageBytesT;
      if (ch * kChunk < unit_nvalid(a, b)) {
        const bool with_q = i == 0 || ch == 0;  // the scoring warps read q on a unit's first item
        mbar_arrive_tx(&full_bar[st], 4 * kBoxBytes + (with_q ? a.G * kD * 2 : 0));
        const int y = u * a.nblk_cap + ch * kChunk;
#pragma unroll
        for (int bx = 0; bx < 4; ++bx) tma_load_2d(sp + bx * kBoxBytes, &tmD, bx * 64, y, &full_bar[st]);
        const __nv_bfloat16* qg = a.q + ((int64_t)b * a.Hq + (int64_t)kvh * a.G) * kD;
        for (int h = 0; h < (with_q ? a.G : 0); ++h)
          asm volatile(
              "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                  smem_u32(sp + 4 * kBoxBytes + h * kQStride * 2)),
              "l"(qg + h * kD), "r"(kD * 2), "r"(smem_u32(&full_bar[st]))
              : "memory");
      } else {
        mbar_arrive(&full_bar[st]);
      }
      issued = i + 1;
    }
    for (int64_t r = 0; r < a.stages && r < issued; ++r) {  // every copy lands before the CTA retires
      const int64_t last = issued - 1 - r;
      if (!mbar_wait(&full_bar[last % a.stages], (uint32_t)((last / a.stages) & 1))) report(a.status, SCOUT_DEV_TIMEOUT);
    }
    return;
  }

  if (warp >= kScoreWarps) {
    // ---------------- selector warps 8..11 -----------------------------------
    const int st = tid - kScoreWarps * 32;
    for (int u = u_first; u <= u_last; ++u) {
      const int e = u - u_first, kb = e & 1;
      uint32_t* keys = keybuf + kb * align4(a.nblk_cap);
      prefetch_unit(a, u, ss);  // overlaps the scoring of u
      if (!mbar_wait(&kfull[kb], (uint32_t)(e >> 1) & 1u) && st == 0) report(a.status, SCOUT_DEV_TIMEOUT);
      const int64_t first = (int64_t)u * a.nchunk, last = first + a.nchunk - 1;
      bool doit = first >= it0 && last < it1;  // the whole unit was scored here
      if (!doit) {
        if (st == 0) {
          const int64_t mine = min(last, it1 - 1) - max(first, it0) + 1;
          __threadfence();  // publish this CTA's scores of u
          const int old = atomicAdd(&a.counters[u], (int)mine);
          s_flag = old + (int)mine == a.nchunk;
          if (s_flag) {
            __threadfence();  // see the other CTAs' scores of u
            a.counters[u] = 0;  // ready for the next call
          }
        }
        sbar();
        doit = s_flag;
        if (doit) {
          const int nvalid = unit_nvalid(a, u / a.Hkv);
          const float* scu = a.scores + (int64_t)u * a.nblk_cap;
          for (int j = st; j < nvalid; j += kSelThreads) keys[j] = score_key(__ldcg(scu + j));
          sbar();
        }
      }
      if (doit) select_unit(a, u, keys, ss);
      if (st == 0) mbar_arrive(&kempty[kb]);  // the key buffer may be refilled
    }
    return;
  }

  // ---------------- scoring warps 0..7 -----------------------------------------
  const int g = lane >> 2, t = lane & 3;
  int ucur = -1, kb = 0;
  bool split = false;
  uint32_t bmm[16][2], bme[8][2];
  for (int64_t i = 0; i < it1 - it0; ++i) {
    const int64_t item = it0 + i;
    const int u = (int)(item / a.nchunk), ch = (int)(item - (int64_t)u * a.nchunk);
    const int nvalid = unit_nvalid(a, u / a.Hkv);
    const int st = (int)(i % a.stages);
    const bool landed = mbar_wait(&full_bar[st], (uint32_t)((i / a.stages) & 1));
    if (!landed && lane == 0) report(a.status, SCOUT_DEV_TIMEOUT);
    const uint8_t* sp = ring + st * kStageBytesT;
    if (u != ucur) {  // the unit's first item in this range
      ucur = u;
      const int e = u - u_first;
      kb = e & 1;
      split = (int64_t)u * a.nchunk < it0 || (int64_t)u * a.nchunk + a.nchunk - 1 >= it1;
      if (!mbar_wait(&kempty[kb], ((uint32_t)(e >> 1) & 1u) ^ 1u) && lane == 0) report(a.status, SCOUT_DEV_TIMEOUT);
      if (ch * kChunk < nvalid && landed) {
        const __nv_bfloat16* qs = reinterpret_cast<const __nv_bfloat16*>(sp + 4 * kBoxBytes);
        if (KIND == SCOUT_DIGEST_MINMAX) {
          minmax_b_frag(qs, a.G, lane, bmm);
        } else {
          mean_b_frag(qs, a.G, lane, bme);
        }
      }
    }
    const int j0 = ch * kChunk + warp * 16;
    if (j0 < a.nblk_cap) {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      if (j0 < nvalid && landed) score_tile<KIND>(smem_u32(sp), warp * 16, lane, bmm, bme, c);
      // pool over the heads of the group (columns 2t, 2t+1 < G), then across t
      const float ninf = -INFINITY;
      float m0 = fmaxf(2 * t < a.G ? c[0] : ninf, 2 * t + 1 < a.G ? c[1] : ninf);
      float m1 = fmaxf(2 * t < a.G ? c[2] : ninf, 2 * t + 1 < a.G ? c[3] : ninf);
      m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
      m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
      if (t == 0) {
        const int r0 = j0 + g, r1 = j0 + g + 8;
        uint32_t* keys = keybuf + kb * align4(a.nblk_cap);
        if (r0 < nvalid) keys[r0] = score_key(m0);
        if (r1 < nvalid) keys[r1] = score_key(m1);
        if (a.user_scores || split) {
          float* scu = a.scores + (int64_t)u * a.nblk_cap;
          if (r0 < a.nblk_cap) scu[r0] = r0 < nvalid ? m0 : ninf;
          if (r1 < a.nblk_cap) scu[r1] = r1 < nvalid ? m1 : ninf;
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&empty_bar[st]);
      if (ch == a.nchunk - 1 || i == it1 - it0 - 1) mbar_arrive(&kfull[kb]);  // this warp's keys of u are in
    }
  }
}

inline size_t counters_bytes(int64_t units) { return (size_t)((units * 4 + 255) / 256 * 256); }

}  // namespace
}  // namespace scout

extern "C" size_t scout_score_topk_workspace_bytes(int B, int Hkv, int nblk_cap) {
  if (B <= 0 || Hkv <= 0 || nblk_cap <= 0) return 0;
  const int64_t units = (int64_t)B * Hkv;
  return scout::counters_bytes(units) + (size_t)units * nblk_cap * sizeof(float);
}

extern "C" int scout_score_topk(int kind, const void* q, const void* digest, const int32_t* seq_len,
                                const uint32_t* resident_bits, const int32_t* prev_cpu_list,
                                const int32_t* prev_cpu_count, int B, int Hq, int Hkv, int D, int P, int nblk_cap,
                                int k, float* scores, int32_t* topk_idx, int32_t* topk_count, int32_t* res_list,
                                int32_t* res_count, int32_t* cpu_list, int32_t* cpu_count, int32_t* delta_list,
                                int32_t* delta_count, void* workspace, size_t workspace_bytes,
                                const scout_launch* launch, cudaStream_t stream) {
  using namespace scout;
  if (q == nullptr || digest == nullptr || seq_len == nullptr || resident_bits == nullptr || topk_idx == nullptr ||
      topk_count == nullptr || res_list == nullptr || res_count == nullptr || cpu_list == nullptr ||
      cpu_count == nullptr || delta_list == nullptr || delta_count == nullptr)
    return SCOUT_ERR_INVALID_ARG;
  if ((prev_cpu_list == nullptr) != (prev_cpu_count == nullptr)) return SCOUT_ERR_INVALID_ARG;
  if (launch != nullptr && launch->max_ctas < 0) return SCOUT_ERR_INVALID_ARG;
  if (kind != SCOUT_DIGEST_MINMAX && kind != SCOUT_DIGEST_MEAN) return SCOUT_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || nblk_cap <= 0 || k <= 0) return SCOUT_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  const int64_t units = (int64_t)B * Hkv;
  if (D != kD || !valid_P(P) || G > kMaxG || nblk_cap > kMaxNblk || units * nblk_cap > 0x7fffffffLL ||
      !aligned16(digest) || !aligned16(q))
    return SCOUT_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < scout_score_topk_workspace_bytes(B, Hkv, nblk_cap))
    return SCOUT_ERR_WORKSPACE;
  TopkArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.digest = static_cast<const uint8_t*>(digest);
  a.seq_len = seq_len;
  a.resident_bits = resident_bits;
  a.prev_list = prev_cpu_list;
  a.prev_count = prev_cpu_count;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = G;
  a.P = P;
  a.nblk_cap = nblk_cap;
  a.k = k;
  a.words = (nblk_cap + 31) / 32;
  a.nchunk = (nblk_cap + kChunk - 1) / kChunk;
  a.n_items = units * a.nchunk;
  a.counters = static_cast<int32_t*>(workspace);
  a.status = nullptr;
  a.user_scores = scores != nullptr;
  a.scores = scores != nullptr ? scores
                               : reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + counters_bytes(units));
  a.topk_idx = topk_idx;
  a.topk_count = topk_count;
  a.res_list = res_list;
  a.res_count = res_count;
  a.cpu_list = cpu_list;
  a.cpu_count = cpu_count;
  a.delta_list = delta_list;
  a.delta_count = delta_count;
  // the digest as a 2-D bf16 tensor [units * nblk_cap rows][256 columns] (512-byte rows
  // for both kinds); 128-row x 64-column boxes with the 128-byte swizzle
  CUtensorMap tmD;
  {
    const cuuint64_t dims[2] = {256, (cuuint64_t)units * nblk_cap};
    const cuuint64_t strides[1] = {512};
    const cuuint32_t box[2] = {64, (cuuint32_t)kChunk};
    const cuuint32_t estr[2] = {1, 1};
    if (encode_tiled(&tmD, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(digest), dims, strides, box, estr,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return SCOUT_ERR_UNSUPPORTED;
  }
  const size_t keys_bytes = (size_t)(2 * align4(nblk_cap) + 2 * align4(a.words) + kBins) * sizeof(uint32_t);
  // per-block limit 232448 bytes (227 KiB) covers static (< 512 bytes here) and dynamic shared memory
  const size_t budget = 232448 - 512 - 1024 - keys_bytes;
  a.stages = (int)min((size_t)kMaxStagesT, budget / kStageBytesT);
  const size_t smem = 1024 + (size_t)a.stages * kStageBytesT + keys_bytes;
  auto kern = kind == SCOUT_DIGEST_MINMAX ? score_topk_kernel<SCOUT_DIGEST_MINMAX> : score_topk_kernel<SCOUT_DIGEST_MEAN>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
    return SCOUT_ERR_CUDA;
  const int cap = launch != nullptr && launch->max_ctas > 0 ? launch->max_ctas : sm_count();
  const int grid = (int)(a.n_items < (int64_t)cap ? a.n_items : (int64_t)cap);  // <= one CTA per item
  kern<<<grid, kThreadsAll, smem, stream>>>(tmD, a);
  return launch_status();
}

// ---------------------------------------------------------------------------
// Allocation-free variant of scout_score_topk.
//
// Some callers cannot allocate device memory at the point where they select
// blocks: engines that reserve all GPU memory in one pool at start-up and forbid
// later cudaMalloc calls (a cudaMalloc can stall other streams and fragment the
// pool), or hosts that load this library as a plugin and hand it no allocator.
// For them the scratch lives in one file-scope device array of fixed size that
// every GPU loading the library keeps until the process exits.
// ---------------------------------------------------------------------------
namespace scout {
namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;  // 4 MiB: counters + fp32 scores
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) uint8_t g_topk_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kNoAllocMaxDevices] = {};

// Device address of g_topk_scratch on the current device, looked up once per
// device (the host-side symbol is only a stand-in and must never reach a kernel).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SCOUT_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return SCOUT_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess || p == nullptr) return SCOUT_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SCOUT_OK;
}

}  // namespace
}  // namespace scout

extern "C" size_t scout_score_topk_noalloc_max_bytes(void) { return scout::kNoAllocScratchBytes; }

extern "C" int scout_score_topk_noalloc(int kind, const void* q, const void* digest, const int32_t* seq_len,
                                        const uint32_t* resident_bits, const int32_t* prev_cpu_list,
                                        const int32_t* prev_cpu_count, int B, int Hq, int Hkv, int D, int P,
                                        int nblk_cap, int k, float* scores, int32_t* topk_idx, int32_t* topk_count,
                                        int32_t* res_list, int32_t* res_count, int32_t* cpu_list, int32_t* cpu_count,
                                        int32_t* delta_list, int32_t* delta_count, cudaStream_t stream) {
  using namespace scout;
  const size_t need = scout_score_topk_workspace_bytes(B, Hkv, nblk_cap);
  if (need == 0) return SCOUT_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return SCOUT_ERR_WORKSPACE;  // beyond the fixed scratch
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != SCOUT_OK) return rc;
  // the array keeps whatever the previous call left: zero the per-unit counters
  if (cudaMemsetAsync(scratch, 0, counters_bytes((int64_t)B * Hkv), stream) != cudaSuccess) return SCOUT_ERR_CUDA;
  return scout_score_topk(kind, q, digest, seq_len, resident_bits, prev_cpu_list, prev_cpu_count, B, Hq, Hkv, D, P,
                          nblk_cap, k, scores, topk_idx, topk_count, res_list, res_count, cpu_list, cpu_count,
                          delta_list, delta_count, scratch, kNoAllocScratchBytes, nullptr, stream);
}
